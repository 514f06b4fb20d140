"""The float64 oracle pinned to what the pages and mathematics fix (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

from oracle import exact
from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import workloads as W
from tests import oracle_pins as pins


def test_exact_fraction_enumeration_matches_page():
    """Exact fractions reproduce every number the worked example prints, and the wrong
    're-sample from p' branch gives (0.35, 0.39, 0.26)."""
    G = pins.golden("three_token_example.json")
    law = exact.one_step_law(pins.frac_list(G["p"]), pins.frac_list(G["q"]))
    assert law["accept_prob"] == pins.frac_list(G["accept_prob"])
    assert law["accepted"] == pins.frac_list(G["accepted_mass"])
    assert sum(law["accepted"]) == Fraction(G["accepted_total"])
    assert law["reject"] == Fraction(G["reject_mass"])
    assert law["residual_unnormalised"] == pins.frac_list(G["residual_unnormalised"])
    assert law["residual"] == pins.frac_list(G["residual"])
    assert law["output"] == pins.frac_list(G["output"])
    wrong = exact.one_step_law(pins.frac_list(G["p"]), pins.frac_list(G["q"]), residual="p")
    assert wrong["output"] == pins.frac_list(G["wrong_variant_output"])


def test_float64_oracle_three_token_example():
    out = pins.check_three_token_example()
    G = pins.golden("three_token_example.json")
    law = exact.one_step_law(pins.frac_list(G["p"]), pins.frac_list(G["q"]))
    assert np.allclose(out, [float(x) for x in law["output"]], atol=1e-15, rtol=0)


def test_greedy_tables():
    pins.check_greedy_tables()


def test_expected_tokens_closed_form():
    pins.check_expected_tokens()


@pytest.mark.parametrize("V,gamma,T,seed,zero", [(3, 1, 1.0, 1, 0.0), (3, 2, 0.7, 2, 0.0),
                                                  (4, 2, 1.3, 3, 0.3), (2, 3, 1.0, 4, 0.0)])
def test_joint_law_brute_force(V, gamma, T, seed, zero):
    pins.check_joint_law(V, gamma, T, seed, zero_frac=zero)


def test_inverse_cdf_convention():
    pins.check_inverse_cdf_convention()


def test_greedy_tie_rule():
    pins.check_greedy_tie_rule()


def test_residual_plus_kept_mass_is_p():
    """min(p, q) + R r = p for every id (tutorial §7.2), on random rows."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        V = int(rng.integers(2, 60))
        p = O.softmax_at_temperature(rng.normal(0, 2, V), 0.9)
        q = O.softmax_at_temperature(rng.normal(0, 2, V), 0.9)
        w = O.residual_weights(p, q)
        R = w.sum()
        assert abs(R - (1 - np.minimum(p, q).sum())) < 1e-14
        assert np.allclose(np.minimum(p, q) + R * (w / R), p, atol=1e-15)


def test_chi_square_three_token_trials():
    """1e5 seeded trials of the worked example (generator's three-token batch): the first
    emitted token follows p; the planted 're-sample from p' mistake is rejected."""
    wl = W.three_token_workload(100_000, seed=0)
    p = np.array([0.5, 0.3, 0.2])

    def first_tokens():
        res = O.verify_batch(wl.target, wl.draft, "f32", wl.draft_tokens, wl.num_draft,
                             wl.temperature, wl.u_accept, wl.u_sample)
        return np.bincount([r.tokens[0] for r in res], minlength=3)

    counts = first_tokens()
    assert stats.chisquare(counts, p * counts.sum()).pvalue > 1e-3, counts
    saved = O.residual_weights
    try:
        O.residual_weights = lambda pp, qq: pp.copy()
        bad = first_tokens()
    finally:
        O.residual_weights = saved
    assert stats.chisquare(bad, p * bad.sum()).pvalue < 1e-6, bad


def test_special_cases():
    # V = 1: the only token is always kept and the bonus is that token
    P = np.zeros((4, 1))
    Q = np.zeros((3, 1))
    r = O.verify_sample_sequence(P, Q, np.zeros(3, int), 3, 1.0, np.full(3, 0.999), 0.999)
    assert r.m == 3 and r.tokens == [0, 0, 0, 0] and r.status == 0
    # q == p: r = 1, every draft kept whatever u in [0,1); no NaN anywhere
    rng = np.random.default_rng(5)
    P = rng.normal(0, 3, (5, 40))
    Q = P[:4].copy()
    r = O.verify_sample_sequence(P, Q, np.array([3, 7, 1, 0]), 4, 0.8,
                                 np.full(4, np.nextafter(np.float32(1), np.float32(0))), 0.3)
    assert r.m == 4 and r.status == 0 and all(np.isfinite(r.p_draft))
    # an out-of-range draft is a rejection (bit 1); with q == p the residual is empty, so
    # the correction falls back to p_m (bit 2) instead of dividing by R = 0
    r = O.verify_sample_sequence(P, Q, np.array([3, 40, 1, 0]), 4, 0.8, np.zeros(4), 0.3)
    assert r.m == 1 and r.status == (O.ST_BAD_DRAFT | O.ST_R_ZERO) and r.mass == 0.0
    p1 = O.softmax_at_temperature(P[1], 0.8)
    assert r.tokens[-1] == int(np.flatnonzero(np.cumsum(p1) > 0.3 * np.cumsum(p1)[-1])[0])
    # a draft the target gives zero probability is never kept, even with u = 0
    P2 = np.log(np.array([[0.5, 0.5, 0.0], [0.2, 0.3, 0.5]]))
    Q2 = np.log(np.array([[0.2, 0.3, 0.5]]))
    r = O.verify_sample_sequence(P2, Q2, np.array([2]), 1, 1.0, np.zeros(1), 0.0)
    assert r.m == 0 and r.tokens == [0]
    # temperature <= 0 selects greedy verification; num_draft is clamped into [0, gmax]
    tgt = W.f32_to_bf16_bits(rng.normal(0, 3, (2, 4, 16)).astype(np.float32))
    drf = W.f32_to_bf16_bits(rng.normal(0, 3, (2, 3, 16)).astype(np.float32))
    toks = np.zeros((2, 3), np.int32)
    res = O.verify_batch(tgt, drf, "bf16", toks, np.array([9, -2]), np.array([0.0, 1.0]),
                         np.zeros((2, 3)), np.zeros(2))
    assert res[0].greedy and res[0].gamma == 3 and res[0].status & O.ST_CLAMPED_GAMMA
    assert (not res[1].greedy) and res[1].gamma == 0 and res[1].m == 0
    assert res[1].status == O.ST_CLAMPED_GAMMA
    # gamma = 0 is a plain decode step: one token sampled from row 0
    p0 = O.softmax_at_temperature(O.widen(tgt[1, 0], "bf16"), 1.0)
    assert res[1].tokens == [int(np.flatnonzero(np.cumsum(p0) > 0)[0])]


def test_commit_kv_lengths():
    """Trim to t+m, then t+m+1 once the new token is processed (tutorial §5.2)."""
    t = np.array([100, 7, 0])
    m = np.array([2, 0, 4])
    kv, dkv, _, _, st = O.commit_kv_lengths(t, m, False, draft_kv_len=t)
    assert list(kv) == [102, 7, 4] and list(dkv) == [102, 7, 4] and not st.any()
    kv, _, _, _, _ = O.commit_kv_lengths(t, m, True)
    assert list(kv) == [103, 8, 5]
    out = np.array([[5, 6, 9, -1, -1], [4, -1, -1, -1, -1], [1, 2, 3, 4, 8]])
    hist = np.full((3, 6), -1)
    clen = np.array([1, 0, 3])
    kv, _, hist2, clen2, st = O.commit_kv_lengths(t, m, True, out_tokens=out, history=hist,
                                                  committed_len=clen)
    assert list(clen2) == [4, 1, 3] and list(st) == [0, 0, O.ST_HISTORY_FULL]
    assert list(hist2[0]) == [-1, 5, 6, 9, -1, -1] and list(hist2[1]) == [4, -1, -1, -1, -1, -1]
    assert list(kv) == [103, 8, 0]          # the overflowing sequence is left untouched
    # a negative committed length is not a legal append position either
    kv, _, hist3, clen3, st = O.commit_kv_lengths(t, m, True, out_tokens=out, history=hist,
                                                  committed_len=np.array([-1, 0, 0]))
    assert list(st) == [O.ST_HISTORY_FULL, 0, 0] and list(kv) == [100, 8, 5]
    assert list(clen3) == [-1, 1, 5] and (hist3[0] == -1).all()


def test_greedy_workload_closed_form():
    """Planted greedy workload: P(m = j) = a^j (1-a), E[emitted] = (1-a^6)/(1-a) = 3.68928
    at a = 0.8, gamma = 5 (closed form of the tutorial §8 and the seventnews article)."""
    wl = W.greedy_32k(seed=0)
    res = O.verify_batch(wl.target, None, "bf16", wl.draft_tokens, wl.num_draft, None, None, None)
    L = np.array([len(r.tokens) for r in res], dtype=float)
    a, g = 0.8, 5
    mean = (1 - a ** (g + 1)) / (1 - a)
    var = sum((j + 1) ** 2 * a ** j * (1 - a) for j in range(g)) + (g + 1) ** 2 * a ** g - mean ** 2
    assert abs(L.mean() - mean) < 4 * np.sqrt(var / len(L)), L.mean()
    # every greedy step emits the planted argmax at the stopping row
    for b, r in enumerate(res):
        row = W.bf16_bits_to_f32(wl.target[b, r.m])
        assert r.tokens[-1] == int(np.argmax(row))


def test_stops_match_step_by_step_decoding():
    """Speculative rounds (oracle verify + stops) reproduce greedy step-by-step decoding that
    ends at the first end token or at the length limit ([TUT] §12.3, §5.2)."""
    pins.check_stops_match_step_by_step()


def test_stops_special_cases():
    out = np.array([[5, 0, 7, 9], [4, 6, -1, -1], [1, 2, 3, 4], [0, 8, 8, 8]])
    m = np.array([3, 1, 3, 3])
    o, mm, st = O.apply_stops(out, m, 0, None)
    assert o.tolist() == [[5, 0, -1, -1], [4, 6, -1, -1], [1, 2, 3, 4], [0, -1, -1, -1]]
    assert mm.tolist() == [1, 1, 3, 0] and st.tolist() == [O.ST_STOPPED, 0, 0, O.ST_STOPPED]
    # budgets: 2 cuts a block (and stops), 5 does not bind, 0 emits nothing, -3 too
    o, mm, st = O.apply_stops(out, m, -1, np.array([2, 5, 0, -3]))
    assert o.tolist() == [[5, 0, -1, -1], [4, 6, -1, -1], [-1] * 4, [-1] * 4]
    assert mm.tolist() == [1, 1, 0, 0] and st.tolist() == [O.ST_STOPPED, 0, O.ST_STOPPED, O.ST_STOPPED]
    # a budget that lands exactly on the emit length stops the sequence, one above does not
    o, mm, st = O.apply_stops(out, m, -1, np.array([4, 3, 4, 5]))
    assert st.tolist() == [O.ST_STOPPED, 0, O.ST_STOPPED, 0] and mm.tolist() == [3, 1, 3, 3]
    # commit appends only the emitted tokens of a cut round
    kv, _, hist, clen, st = O.commit_kv_lengths(np.array([10, 10]), np.array([0, 1]), False,
                                                out_tokens=np.array([[-1, -1], [4, 6]]),
                                                history=np.full((2, 4), -9), committed_len=np.array([1, 1]))
    assert clen.tolist() == [1, 3] and hist.tolist() == [[-9] * 4, [-9, 4, 6, -9]] and kv.tolist() == [10, 11]


def test_tree_figure():
    pins.check_tree_figure()


def test_tree_chain_equals_chain_verification():
    pins.check_tree_chain_equals_chain()


def test_tree_matches_target_greedy_walk():
    pins.check_tree_matches_greedy_walk()


def test_tree_ties_and_invalid_nodes():
    pins.check_tree_ties_and_invalid_nodes()


def test_tree_batch_clamps_node_counts():
    rows = np.zeros((2, 3, 4), dtype=np.float32)
    rows[:, 0, 1] = 1.0
    rows[:, 1, 2] = 1.0
    res = O.verify_tree_batch(rows, "f32", np.array([[1, 2], [1, 3]]), np.array([[0, 1], [0, 1]]),
                              np.array([5, -1]))
    assert res[0].n == 2 and res[0].status == O.ST_CLAMPED_GAMMA and res[0].tokens == [1, 2, 0]
    assert res[1].n == 0 and res[1].status == O.ST_CLAMPED_GAMMA and res[1].tokens == [1]


def test_truncation_against_counting():
    pins.check_truncation_against_counting()


def test_top_k_one_is_greedy():
    pins.check_top_k_one_is_greedy()


def test_truncation_off_switches():
    pins.check_truncation_off_switches()


@pytest.mark.parametrize("V,gamma,T,k,tp,seed", [(4, 2, 1.0, 2, 1.0, 31), (4, 2, 0.8, 0, 0.7, 32),
                                                  (4, 1, 1.3, 3, 0.6, 33), (3, 2, 1.0, 2, 0.9, 34)])
def test_truncated_joint_law(V, gamma, T, k, tp, seed):
    pins.check_truncated_joint_law(V, gamma, T, k, tp, seed)


def test_accept_margin_is_distance_to_decision_flip():
    pins.check_accept_margin()


def test_inverse_cdf_margin_is_distance_to_token_change():
    pins.check_inverse_cdf_margin()


def test_top_p_margin_is_distance_to_kept_set_change():
    pins.check_top_p_margin()


def test_flagged_uses_every_margin():
    pins.check_flagged_uses_every_margin()



def test_rows_without_a_distribution_are_marked():
    pins.check_rows_without_distribution()


def test_truncated_entry_masks_nan_logits():
    pins.check_truncated_entry_masks_nan()
