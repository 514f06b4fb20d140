"""Stops on the GPU (spec_apply_stops, and commit of a cut round) against the oracle: bit-exact
on seeded synthetic rounds, and as the last stage of a greedy verify pipeline."""
import numpy as np
import pytest
import torch

from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests.parity import dev, oracle_results, run_gpu

pytestmark = pytest.mark.gpu


def _rounds(B, g, vocab, seed):
    """Seeded synthetic rounds: m uniform in [0, g] (plus out-of-range values that clamp),
    emitted tokens drawn from a small vocabulary so that end tokens recur, -1 after the emit."""
    rng = np.random.default_rng([2026, 40, seed])
    m = rng.integers(0, g + 1, B).astype(np.int32)
    m[:3] = [-2, g + 5, 0]
    out = np.full((B, g + 1), -1, np.int32)
    for b in range(B):
        n = int(np.clip(m[b], 0, g)) + 1
        out[b, :n] = rng.integers(0, vocab, n)
    return out, m, rng


@pytest.mark.parametrize("g", [0, 1, 4, 32])
def test_apply_stops_matches_oracle(g):
    B = 517
    out, m, rng = _rounds(B, g, 6, g)
    budgets = rng.integers(-2, g + 4, B).astype(np.int32)
    for eos, use_budget in [(0, False), (-1, True), (3, True), (5, False), (-1, False)]:
        O_ = dev(out)
        M_ = dev(m)
        S_ = dev(np.full(B, 64, np.int32))          # existing bits are kept
        N_ = dev(budgets) if use_budget else None
        sv.spec_apply_stops(O_, M_, eos, N_, S_)
        torch.cuda.synchronize()
        wo, wm, ws = O.apply_stops(out, m, eos, budgets if use_budget else None)
        assert np.array_equal(O_.cpu().numpy(), wo), (g, eos, use_budget)
        assert np.array_equal(M_.cpu().numpy(), wm), (g, eos, use_budget)
        assert np.array_equal(S_.cpu().numpy(), ws | 64), (g, eos, use_budget)


def test_verify_stops_commit_pipeline_greedy():
    """Greedy verify -> stops -> commit with history, on the GPU and in the oracle, from the
    same workload; the end token is the id the targets emit most often."""
    wl = W.greedy_32k(seed=3)
    B, g = wl.B, wl.gmax
    gpu = run_gpu(wl)
    res = oracle_results(wl)
    want_out = O.emitted_rows(res, g)
    want_m = np.array([r.m for r in res])
    assert np.array_equal(gpu["out"], want_out) and np.array_equal(gpu["m"], want_m)
    ids, counts = np.unique(want_out[want_out >= 0], return_counts=True)
    eos = int(ids[np.argmax(counts)])
    budgets = np.random.default_rng([2026, 41]).integers(1, g + 3, B).astype(np.int32)
    O_, M_, S_ = dev(gpu["out"]), dev(gpu["m"]), dev(np.zeros(B, np.int32))
    sv.spec_apply_stops(O_, M_, eos, dev(budgets), S_)
    cap = 64
    t = np.random.default_rng([2026, 42]).integers(512, 8193, B).astype(np.int32)
    hist = np.full((B, cap), -1, np.int32)
    clen = np.zeros(B, np.int32)
    T_, H_, C_ = dev(t), dev(hist), dev(clen)
    sv.spec_commit_kv_lengths(M_, T_, None, False, O_, H_, C_, S_)
    torch.cuda.synchronize()
    so, sm, ss = O.apply_stops(want_out, want_m, eos, budgets)
    kv, _, hh, cc, cs = O.commit_kv_lengths(t, sm, False, out_tokens=so, history=hist, committed_len=clen)
    assert np.array_equal(O_.cpu().numpy(), so) and np.array_equal(M_.cpu().numpy(), sm)
    assert np.array_equal(S_.cpu().numpy(), ss | cs)
    assert np.array_equal(T_.cpu().numpy(), kv) and np.array_equal(H_.cpu().numpy(), hh)
    assert np.array_equal(C_.cpu().numpy(), cc)
    assert (ss & O.ST_STOPPED).any() and not (ss & O.ST_STOPPED).all()
