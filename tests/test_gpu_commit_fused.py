"""The fused verify-and-commit calls leave exactly what the verify call followed by
spec_commit_kv_lengths leaves: tokens, accepted counts, diag, status (history overflow
included), both KV lengths, the history and the committed lengths."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests.parity import dev

pytestmark = pytest.mark.gpu


def _state(wl, cap, seed):
    rng = np.random.default_rng(seed)
    B = wl.B
    clen = rng.integers(0, cap, B).astype(np.int32)
    clen[::7] = cap - 1            # no room for a whole round: left untouched, flagged
    clen[3] = -1                   # an illegal append position: likewise
    hist = np.full((B, cap), -5, np.int32)
    t = wl.kv_len.astype(np.int32)
    return {"t": dev(t), "d": dev(t + 1), "h": dev(hist), "c": dev(clen)}


def _outs(wl):
    B, g = wl.B, wl.gmax
    return (torch.full((B, g + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, 2 * g + 1), 1.5, dtype=torch.float32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"))


def _host(*ts):
    return [t.cpu().numpy() for t in ts]


@pytest.mark.parametrize("name", ["sampling", "mixed", "greedy", "truncated"])
def test_fused_commit_equals_separate_calls(name):
    if name == "sampling":
        wl = W.sampling_workload("fused-s", cfg=61, seed=0, B=96, gmax=4, V=128256, dtype="bf16",
                                 target_sigma=3.0, draft_scale=0.7, draft_sigma=1.0, temperature=0.8)
    elif name == "mixed":
        wl = W.sampling_workload("fused-m", cfg=62, seed=0, B=64, gmax=6, V=50000, dtype="f32",
                                 target_sigma=3.0, draft_scale=1.0, draft_sigma=1.5, temperature=0.7,
                                 num_draft=np.arange(64) % 7, greedy_mask=(np.arange(64) % 2) == 0)
    elif name == "truncated":
        wl = W.sampling_workload("fused-t", cfg=64, seed=0, B=48, gmax=4, V=40000, dtype="bf16",
                                 target_sigma=3.0, draft_scale=0.8, draft_sigma=1.0, temperature=0.9,
                                 num_draft=np.arange(48) % 5, greedy_mask=(np.arange(48) % 6) == 0)
    else:
        wl = W.greedy_planted_workload("fused-g", cfg=63, seed=0, B=64, gmax=5, V=32000, alpha=0.8)
    trunc = name == "truncated"
    tk = dev(np.where(np.arange(wl.B) % 3 == 0, 0, 40).astype(np.int32))
    tp = dev(np.where(np.arange(wl.B) % 4 == 1, 1.0, 0.85).astype(np.float32))
    cap = 12
    code = sv.SPEC_BF16 if wl.dtype == "bf16" else sv.SPEC_F32
    ws = torch.zeros(sv.spec_verify_workspace_bytes(wl.B, wl.gmax, wl.V, code), dtype=torch.uint8, device="cuda")
    tgt, toks, nd = dev(wl.target), dev(wl.draft_tokens), dev(wl.num_draft)
    got = {}
    for fused in (False, True):
        for proc in (True, False):
            st = _state(wl, cap, seed=5)
            out, m, dg, status = _outs(wl)
            if wl.greedy_only:
                if fused:
                    sv.spec_verify_greedy_commit(tgt, toks, nd, out, m, st["t"], st["d"], proc, st["h"], st["c"],
                                                 status=status, workspace=ws)
                else:
                    sv.spec_verify_greedy(tgt, toks, nd, out, m, status, workspace=ws)
                    sv.spec_commit_kv_lengths(m, st["t"], st["d"], proc, out, st["h"], st["c"], status)
            else:
                args = (tgt, dev(wl.draft), toks, nd, dev(wl.temperature), dev(wl.u_accept), dev(wl.u_sample),
                        out, m)
                targs = (tgt, dev(wl.draft), toks, nd, dev(wl.temperature), tk, tp, dev(wl.u_accept),
                         dev(wl.u_sample), out, m)
                if trunc and fused:
                    sv.spec_verify_sample_truncated_commit(*targs, st["t"], st["d"], proc, st["h"], st["c"],
                                                           diag=dg, status=status, workspace=ws)
                elif trunc:
                    sv.spec_verify_sample_truncated(*targs, diag=dg, status=status, workspace=ws)
                    sv.spec_commit_kv_lengths(m, st["t"], st["d"], proc, out, st["h"], st["c"], status)
                elif fused:
                    sv.spec_verify_sample_commit(*args, st["t"], st["d"], proc, st["h"], st["c"], diag=dg,
                                                 status=status, workspace=ws)
                else:
                    sv.spec_verify_sample(*args, diag=dg, status=status, workspace=ws)
                    sv.spec_commit_kv_lengths(m, st["t"], st["d"], proc, out, st["h"], st["c"], status)
            torch.cuda.synchronize()
            got[(fused, proc)] = _host(out, m, dg.view(torch.int32), status, st["t"], st["d"], st["h"], st["c"])
    assert bool((ws == 0).all())
    names = ("out_tokens", "num_accepted", "diag", "status", "target_kv_len", "draft_kv_len", "history",
             "committed_len")
    for proc in (True, False):
        for n, x, y in zip(names, got[(False, proc)], got[(True, proc)]):
            assert np.array_equal(x, y), (name, proc, n)
    status = got[(True, True)][3]
    assert (status & sv.ST_HISTORY_FULL).any() and not (status & sv.ST_HISTORY_FULL).all()


def test_fused_tree_commit_equals_separate_calls():
    """spec_verify_tree_greedy_commit leaves what spec_verify_tree_greedy followed by
    spec_commit_kv_lengths (gmax = nmax) leaves: tokens, path, accepted counts, status, both
    lengths, the history (the path's tokens) and the committed lengths."""
    tw = W.tree_workload("fused-tree", cfg=65, seed=0, B=24, nmax=15, V=32000)
    B, n = tw.B, tw.nmax
    cap = 20
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, n, tw.V, sv.SPEC_BF16), dtype=torch.uint8, device="cuda")
    tgt, toks, pars, nn = dev(tw.target), dev(tw.node_tokens), dev(tw.node_parents), dev(tw.num_nodes)
    got = {}
    for fused in (False, True):
        for proc in (True, False):
            st = _state(tw, cap, seed=6)
            out = torch.full((B, n + 1), -7, dtype=torch.int32, device="cuda")
            m = torch.full((B,), -7, dtype=torch.int32, device="cuda")
            path = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
            status = torch.full((B,), -7, dtype=torch.int32, device="cuda")
            if fused:
                sv.spec_verify_tree_greedy_commit(tgt, toks, pars, nn, out, m, st["t"], st["d"], proc, st["h"],
                                                  st["c"], path_nodes=path, status=status, workspace=ws)
            else:
                sv.spec_verify_tree_greedy(tgt, toks, pars, nn, out, m, path, status, workspace=ws)
                sv.spec_commit_kv_lengths(m, st["t"], st["d"], proc, out, st["h"], st["c"], status, gmax=n)
            torch.cuda.synchronize()
            got[(fused, proc)] = _host(out, m, path, status, st["t"], st["d"], st["h"], st["c"])
    assert bool((ws == 0).all())
    names = ("out_tokens", "num_accepted", "path_nodes", "status", "target_kv_len", "draft_kv_len", "history",
             "committed_len")
    for proc in (True, False):
        for name, x, y in zip(names, got[(False, proc)], got[(True, proc)]):
            assert np.array_equal(x, y), (proc, name)
    # the commit did something: lengths advanced where history had room
    t0 = tw.kv_len.astype(np.int64)
    assert (got[(True, True)][4] != t0).any()
