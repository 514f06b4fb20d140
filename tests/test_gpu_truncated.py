"""Top-k / top-p truncated sampling on the GPU (spec_verify_sample_truncated) against the float64
oracle: tokens and accepted counts bit-exact outside flagged margins (acceptance, inverse CDF
and the top-p crossing), p'(d), q'(d) and the residual mass within 1e-5; workspace returned to
zero; repeat runs bit-identical.  The "M013" card §10 and the nxmr note: truncation must show in
both p and q."""
import math

import numpy as np
import pytest
import torch

from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


def run_truncated(wl, top_k, top_p):
    B, g = wl.B, wl.gmax
    out = torch.full((B, g + 1), -7, dtype=torch.int32, device="cuda")
    m = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    dg = torch.full((B, 2 * g + 1), 1234.5, dtype=torch.float32, device="cuda")
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, g, wl.V, sv.SPEC_BF16), dtype=torch.uint8, device="cuda")
    sv.spec_verify_sample_truncated(parity.dev(wl.target), parity.dev(wl.draft), parity.dev(wl.draft_tokens),
                                    parity.dev(wl.num_draft), parity.dev(wl.temperature),
                                    None if top_k is None else parity.dev(np.asarray(top_k, np.int32)),
                                    None if top_p is None else parity.dev(np.asarray(top_p, np.float32)),
                                    parity.dev(wl.u_accept), parity.dev(wl.u_sample), out, m, dg, st, workspace=ws)
    torch.cuda.synchronize()
    assert bool((ws == 0).all()), "workspace not returned to zero"
    return {"out": out.cpu().numpy(), "m": m.cpu().numpy(), "status": st.cpu().numpy(), "diag": dg.cpu().numpy()}


def check(wl, top_k, top_p, max_differ=1):
    gpu = run_truncated(wl, top_k, top_p)
    res = O.verify_batch(wl.target, wl.draft, wl.dtype, wl.draft_tokens, wl.num_draft, wl.temperature,
                         wl.u_accept, wl.u_sample, top_k=None if top_k is None else np.asarray(top_k),
                         top_p=None if top_p is None else np.asarray(top_p), nan_masked=True)
    n, flagged, differ = parity.compare(wl, gpu, res, check_probs=False)
    parity.record(wl.name, n, flagged, differ, entry="sample_truncated")
    assert len(differ) <= max_differ, (flagged, differ)
    # p'(d_i), q'(d_i) for the drafts the oracle judged
    for b, r in enumerate(res):
        if r.greedy:
            continue
        dg = gpu["diag"][b]
        for i, (pd, qd) in enumerate(zip(r.p_draft, r.q_draft)):
            if not math.isnan(pd) and b not in flagged:
                assert abs(dg[2 * i] - pd) <= parity.PROB_TOL and abs(dg[2 * i + 1] - qd) <= parity.PROB_TOL, \
                    (b, i, dg[2 * i], pd, dg[2 * i + 1], qd)
    return gpu, res


def test_truncation_settings_small_vocabulary():
    B = 16
    wl = W.sampling_workload("trunc-small", cfg=71, seed=0, B=B, gmax=4, V=5000, dtype="bf16",
                             target_sigma=3.0, draft_scale=0.9, draft_sigma=0.7,
                             temperature=[0.8, 1.0, 0.7, 1.2, 0.9, 1.0, 0.6, 1.1, 0.8, 1.0, 0.0, 0.9, 1.0, 0.7, 1.3, 0.8],
                             num_draft=[4, 4, 3, 4, 2, 4, 4, 1, 4, 0, 4, 4, 3, 4, 4, 4],
                             greedy_mask=[0] * 10 + [1] + [0] * 5)
    top_k = [0, 1, 5, 200, 0, 0, 50, 4999, 5000, 30, 20, -3, 3, 100, 0, 1000]
    top_p = [1.0, 1.0, 1.0, 1.0, 0.5, 0.9, 0.8, 0.95, 0.3, 0.7, 0.6, 2.0, 0.99, 0.0, 0.05, 0.999]
    _, res = check(wl, top_k, top_p)
    plain = O.verify_batch(wl.target, wl.draft, wl.dtype, wl.draft_tokens, wl.num_draft, wl.temperature,
                           wl.u_accept, wl.u_sample)
    assert sum(r.tokens != s.tokens for r, s in zip(res, plain)) >= 4   # the truncation matters here


def test_truncation_full_vocabulary():
    wl = W.sampling_workload("trunc-128k", cfg=72, seed=1, B=8, gmax=4, V=128256, dtype="bf16",
                             target_sigma=3.0, draft_scale=0.7, draft_sigma=1.0, temperature=0.8,
                             boost_frac=0.01, boost=8.0)
    check(wl, [50, 50, 0, 0, 1000, 20, 1, 2000], [0.9, 1.0, 0.9, 0.5, 0.95, 0.7, 1.0, 0.8])


def test_ties_at_the_threshold():
    """Logits on a coarse grid: the k-th largest value is shared by many ids, all of them kept."""
    wl = W.sampling_workload("trunc-ties", cfg=73, seed=2, B=10, gmax=3, V=3000, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=0.5, temperature=1.0)
    for arr in (wl.target, wl.draft):
        f = W.bf16_bits_to_f32(arr)
        arr[...] = W.f32_to_bf16_bits(np.round(f))
    check(wl, [1, 2, 7, 40, 300, 5, 1, 60, 3, 10], [1.0, 0.8, 1.0, 0.9, 0.5, 1.0, 0.9, 0.99, 0.6, 1.0])


def test_no_truncation_arrays():
    wl = W.sampling_workload("trunc-off", cfg=74, seed=3, B=6, gmax=5, V=9000, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.9)
    check(wl, None, None)
    check(wl, None, [0.8] * 6)
    check(wl, [64] * 6, None)


def test_repeat_runs_are_bit_identical():
    wl = W.sampling_workload("trunc-repeat", cfg=75, seed=4, B=12, gmax=4, V=20000, dtype="bf16",
                             target_sigma=3.0, draft_scale=0.8, draft_sigma=1.0, temperature=0.8)
    k, p = [40] * 12, [0.9] * 12
    a = run_truncated(wl, k, p)
    b = run_truncated(wl, k, p)
    for key in ("out", "m", "status"):
        assert np.array_equal(a[key], b[key])
    assert np.array_equal(a["diag"].view(np.int32), b["diag"].view(np.int32))


@pytest.mark.parametrize("V", [40000, 151936, 262144, 5001, 270000])
def test_row_layouts(V):
    """Rows that end inside a step of the row pass (V = 40000, 151936, 270000), rows of whole
    steps only (262144 = 16 steps of 16384 ids: no ragged step), and a vocabulary that is not a
    multiple of 8 (5001: the scalar load path, a ragged last vector)."""
    wl = W.sampling_workload(f"trunc-V{V}", cfg=76, seed=5, B=6, gmax=3, V=V, dtype="bf16",
                             target_sigma=3.0, draft_scale=0.8, draft_sigma=1.0,
                             temperature=[0.8, 1.0, 0.0, 0.7, 1.2, 0.9], num_draft=[3, 3, 3, 2, 3, 0],
                             greedy_mask=[0, 0, 1, 0, 0, 0])
    check(wl, [50, 0, 10, 1000, 20, 0], [0.9, 0.8, 1.0, 1.0, 0.5, 0.95])


def test_fused_window_edges():
    """The one-pass search fixes its window from a sample of the row before the pass.  Rows where
    that sample misses the max by far (a planted outlier: the row is searched again from the true
    max), rows of negative logits (windows below zero compare keys), a top-k crossing below both
    fused windows, a low temperature and logits near zero."""
    B = 8
    wl = W.sampling_workload("trunc-fused", cfg=77, seed=6, B=B, gmax=3, V=128256, dtype="bf16",
                             target_sigma=3.0, draft_scale=0.8, draft_sigma=1.0,
                             temperature=[0.8, 1.0, 0.9, 0.05, 1.0, 0.7, 0.8, 1.0], boost_frac=0.01, boost=8.0)
    for arr in (wl.target, wl.draft):
        f = W.bf16_bits_to_f32(arr).astype(np.float32)
        f[0, :, 8003] = 60.0           # id 8003 lies outside the sampled runs
        f[5, :, 77777] = 45.0
        f[1] -= 40.0                   # every logit negative
        f[4] *= 1e-3                   # logits near zero
        arr[...] = W.f32_to_bf16_bits(f)
    check(wl, [50, 0, 40000, 0, 100, 20, 0, 0], [0.9, 0.9, 1.0, 0.9, 0.95, 1.0, 1.0, 0.7])


def test_deep_crossings():
    """Thresholds far below the max in key space (flat logits near zero, where bf16 keys are
    dense; flat negative logits; a top-k of most of the vocabulary): the search narrows the keys
    left to one window in a few passes instead of walking them 256 at a time."""
    B = 6
    wl = W.sampling_workload("trunc-deep", cfg=78, seed=7, B=B, gmax=3, V=128256, dtype="bf16",
                             target_sigma=1.0, draft_scale=0.9, draft_sigma=0.5, temperature=1.0)
    for arr in (wl.target, wl.draft):
        f = W.bf16_bits_to_f32(arr).astype(np.float32)
        f[0:3] *= 1e-3                 # flat, around zero
        f[3:5] = f[3:5] * 1e-2 - 5.0   # flat, negative
        arr[...] = W.f32_to_bf16_bits(f)
    check(wl, [0, 60000, 0, 0, 100000, 127000], [0.9, 1.0, 0.5, 0.95, 0.9, 0.99])


def test_walks_over_empty_keys():
    """Crossings below zero on spread logits: the keys near zero hold few ids or none, and the
    search steps from a window straight to the next key that holds one."""
    wl = W.sampling_workload("trunc-gaps", cfg=80, seed=8, B=4, gmax=2, V=128256, dtype="bf16",
                             target_sigma=3.0, draft_scale=0.9, draft_sigma=0.5, temperature=[5.0, 5.0, 2.0, 1.0])
    check(wl, [0, 125000, 0, 120000], [0.999, 1.0, 0.995, 0.99])


@pytest.mark.parametrize("offset", [0, 1])
def test_split_layout_matches_one_array(offset):
    """spec_verify_sample_truncated_split (target row 0 in an array of its own) gives the
    one-array call's bits, on the 128-bit path and (offset 1: misaligned) the scalar path, and
    with gmax = 0."""
    for gmax in (4, 0):
        wl = W.sampling_workload(f"trunc-split-{gmax}", cfg=81, seed=9 + offset, B=6, gmax=gmax, V=20000,
                                 dtype="bf16", target_sigma=3.0, draft_scale=0.8, draft_sigma=1.0,
                                 temperature=[0.8, 1.0, 0.0, 0.7, 1.2, 0.9],
                                 greedy_mask=[0, 0, 1, 0, 0, 0])
        k = np.asarray([50, 0, 10, 1000, 20, 0], np.int32)
        p = np.asarray([0.9, 0.8, 1.0, 1.0, 0.5, 0.95], np.float32)
        one = run_truncated(wl, k, p)
        tgt = parity.dev(wl.target)
        B, g, V = wl.B, wl.gmax, wl.V

        def place(t):
            if offset == 0:
                return t.contiguous()
            buf = torch.empty(t.numel() + offset, dtype=t.dtype, device=t.device)
            view = buf[offset:].view(t.shape)
            view.copy_(t)
            return view

        saved = place(tgt[:, 0, :])
        block = place(tgt[:, 1:, :]) if g > 0 else None
        out = torch.full((B, g + 1), -7, dtype=torch.int32, device="cuda")
        m = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        dg = torch.full((B, 2 * g + 1), 1234.5, dtype=torch.float32, device="cuda")
        st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        ws = torch.zeros(sv.spec_verify_workspace_bytes(B, g, V, sv.SPEC_BF16), dtype=torch.uint8, device="cuda")
        sv.spec_verify_sample_truncated_split(saved, block, parity.dev(wl.draft), parity.dev(wl.draft_tokens),
                                              parity.dev(wl.num_draft), parity.dev(wl.temperature),
                                              parity.dev(k), parity.dev(p), parity.dev(wl.u_accept),
                                              parity.dev(wl.u_sample), out, m, dg, st, workspace=ws)
        torch.cuda.synchronize()
        assert bool((ws == 0).all())
        assert np.array_equal(out.cpu().numpy(), one["out"]) and np.array_equal(m.cpu().numpy(), one["m"])
        assert np.array_equal(st.cpu().numpy(), one["status"])
        assert np.array_equal(dg.cpu().numpy().view(np.int32), one["diag"].view(np.int32))
