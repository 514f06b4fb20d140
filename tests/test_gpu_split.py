"""The split layout (target row 0 in an array of its own, rows 1..gmax in another) gives
bit-identical results to the one-array layout, and so the oracle's, on greedy, sampling and
mixed batches, fp32 and bf16, the 128-bit and the scalar load paths, and gmax = 0.

Tutorial "投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡", §4: row 0 of the alignment table
is the target's prediction saved from the previous round; rows 1..gamma come from this round's
forward over the drafts."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


def _split(target: torch.Tensor, offset_elems: int = 0):
    """saved [B][V] and block [B][gmax][V] copies of a [B][gmax+1][V] target; offset_elems > 0
    places each of them that many elements past an allocation start (misaligned)."""
    B, gp1, V = target.shape

    def place(t):
        if offset_elems == 0:
            return t.contiguous()
        buf = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device=t.device)
        view = buf[offset_elems:].view(t.shape)
        view.copy_(t)
        return view

    saved = place(target[:, 0, :])
    block = place(target[:, 1:, :]) if gp1 > 1 else None
    return saved, block


def _outs(B, g):
    return (torch.full((B, g + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, 2 * g + 1), 1234.5, dtype=torch.float32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"))


def _run(wl, split: bool, greedy: bool, offset_elems: int = 0):
    B, g = wl.B, wl.gmax
    tgt = parity.dev(wl.target)
    toks, nd = parity.dev(wl.draft_tokens), parity.dev(wl.num_draft)
    out, m, dg, st = _outs(B, g)
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, g, wl.V, sv.SPEC_BF16 if wl.dtype == "bf16" else sv.SPEC_F32),
                     dtype=torch.uint8, device="cuda")
    if split:
        saved, block = _split(tgt, offset_elems)
        if greedy:
            sv.spec_verify_greedy_split(saved, block, toks, nd, out, m, st, workspace=ws)
        else:
            sv.spec_verify_sample_split(saved, block, parity.dev(wl.draft), toks, nd, parity.dev(wl.temperature),
                                        parity.dev(wl.u_accept), parity.dev(wl.u_sample), out, m, dg, st,
                                        workspace=ws)
    else:
        if greedy:
            sv.spec_verify_greedy(tgt, toks, nd, out, m, st, workspace=ws)
        else:
            sv.spec_verify_sample(tgt, parity.dev(wl.draft), toks, nd, parity.dev(wl.temperature),
                                  parity.dev(wl.u_accept), parity.dev(wl.u_sample), out, m, dg, st, workspace=ws)
    torch.cuda.synchronize()
    assert bool((ws == 0).all()), "workspace not returned to zero"
    return {"out": out.cpu().numpy(), "m": m.cpu().numpy(), "status": st.cpu().numpy(),
            "diag": None if greedy else dg.cpu().numpy()}


def _same(a, b):
    for k in ("out", "m", "status"):
        assert np.array_equal(a[k], b[k]), k
    if a["diag"] is not None:
        assert np.array_equal(a["diag"].view(np.int32), b["diag"].view(np.int32)), "diag bits"


@pytest.mark.parametrize("dtype,V,offset", [("bf16", 32000, 0), ("bf16", 9000, 1), ("f32", 5003, 0)])
def test_split_sampling_matches_one_array_and_oracle(dtype, V, offset):
    B = 10
    wl = W.sampling_workload("split-sample", cfg=41, seed=1, B=B, gmax=5, V=V, dtype=dtype,
                             target_sigma=3.0, draft_scale=0.8, draft_sigma=1.0,
                             temperature=[0.8, 0.0, 1.1, 0.7, 0.0, 1.0, 0.9, 1.3, 0.6, 0.0],
                             num_draft=[5, 5, 3, 0, 2, 5, 1, 4, 5, 0],
                             greedy_mask=[0, 1, 0, 0, 1, 0, 0, 0, 0, 1])
    one = _run(wl, split=False, greedy=False)
    two = _run(wl, split=True, greedy=False, offset_elems=offset)
    _same(one, two)
    n, flagged, differ = parity.compare(wl, two, parity.oracle_results(wl))
    parity.record(wl.name, n, flagged, differ, entry="sample_split")
    assert n == B and len(differ) <= 1, (flagged, differ)


def test_split_greedy_matches_one_array_and_oracle():
    wl = W.greedy_planted_workload("split-greedy", cfg=42, seed=2, B=24, gmax=5, V=32000, alpha=0.8)
    one = _run(wl, split=False, greedy=True)
    two = _run(wl, split=True, greedy=True)
    _same(one, two)
    n, flagged, differ = parity.compare(wl, two, parity.oracle_results(wl))
    assert n == wl.B and not differ


def test_split_without_drafts_takes_no_block():
    """gmax = 0: every sequence emits its bonus token from the saved row alone."""
    wl = W.sampling_workload("split-g0", cfg=43, seed=3, B=7, gmax=0, V=4096, dtype="bf16",
                             target_sigma=2.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.9)
    one = _run(wl, split=False, greedy=False)
    two = _run(wl, split=True, greedy=False)
    _same(one, two)
    assert (two["m"] == 0).all() and (two["out"][:, 0] >= 0).all()
