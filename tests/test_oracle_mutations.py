"""Plausible mistakes planted in the oracle (on the CPU) must each break at least one pin."""
import numpy as np
import pytest

from oracle import specverify_oracle as O
from tests import oracle_pins as pins


def _shifted_rows(orig):
    # judge draft i with target row i+1 (the tutorial's §4 off-by-one)
    def f(target, draft, drafts, gamma, T, ua, us):
        t2 = np.concatenate([target[1:], target[-1:]], axis=0)
        return orig(t2, draft, drafts, gamma, T, ua, us)
    return f


def _greedy_last_max(row):
    best = np.max(row)
    return int(np.flatnonzero(row == best)[-1])


def _icdf_ge(weights, u):
    C = np.cumsum(weights)
    total = float(C[-1])
    v = int(np.flatnonzero(C >= u * total)[0])
    return v, 1.0, total


def _stops_last_token_only(out_tokens, m, eos_id, max_new=None):
    # the tutorial's loop tests only output[-1] for the end token (an EOS accepted inside the
    # block is emitted and followed by more tokens)
    out = np.array(out_tokens)
    mm = np.array(m)
    st = np.zeros(len(mm), dtype=np.int64)
    for b in range(len(mm)):
        n = int(mm[b]) + 1
        if max_new is not None:
            n = min(n, max(int(max_new[b]), 0))
        if (n >= 1 and out[b, n - 1] == eos_id) or (max_new is not None and n >= int(max_new[b])):
            st[b] |= O.ST_STOPPED
        out[b, n:] = -1
        mm[b] = max(n - 1, 0)
    return out, mm, st


_apply_stops = O.apply_stops


_truncated = O.truncated_distribution
_inverse_cdf = O.inverse_cdf


def _icdf_margin_scaled(f):
    # the inverse CDF with its reported margin scaled by f (the token is unchanged)
    def run(weights, u):
        v, a, total = _inverse_cdf(weights, u)
        return v, a * f, total
    return run


def _top_p_margin_scaled(f):
    # the truncation with its top-p crossing margin scaled by f (the kept set is unchanged)
    def run(logits, T, top_k=0, top_p=1.0):
        d, a = _truncated(logits, T, top_k, top_p)
        return d, a * f
    return run


def _trunc_variant(full_mass=False, strict_k=False):
    # a copy of the truncation with one planted mistake: top-p's target taken over the whole
    # distribution instead of the top-k-kept mass, or top-k dropping the ties at its threshold
    def run(logits, T, top_k=0, top_p=1.0):
        p = O.softmax_at_temperature(logits, T)
        V = len(logits)
        keep = np.ones(V, dtype=bool)
        if 0 < top_k < V:
            tau = np.sort(logits)[::-1][top_k - 1]
            keep &= (logits > tau) if strict_k else (logits >= tau)
            if not keep.any():
                keep[int(np.argmax(logits))] = True
        if 0.0 < top_p < 1.0:
            vals, inv = np.unique(logits[keep], return_inverse=True)
            mass = np.bincount(inv, weights=p[keep], minlength=len(vals))
            cum = np.cumsum(mass[::-1])
            target = top_p * (1.0 if full_mass else float(cum[-1]))
            hits = np.flatnonzero(cum >= target)
            j = int(hits[0]) if hits.size else len(cum) - 1
            keep &= logits >= vals[::-1][j]
        w = np.where(keep, p, 0.0)
        return w / np.sum(w), np.inf
    return run


def _tree_variant(own_row=False, last_tie=False):
    # a copy of the tree verification with one planted mistake: the node's own row judged
    # instead of its parent's, or the higher index winning equal depths
    def run(target, node_tokens, node_parents, n):
        V = target.shape[1]
        status, acc, depth, best = 0, [True] + [False] * n, [0] * (n + 1), 0
        for j in range(1, n + 1):
            par, d = int(node_parents[j - 1]), int(node_tokens[j - 1])
            if not (0 <= par < j):
                status |= O.ST_BAD_TREE
                continue
            depth[j] = depth[par] + 1
            if not acc[par]:
                continue
            if not (0 <= d < V):
                status |= O.ST_BAD_DRAFT
                continue
            row = target[j] if own_row else target[par]
            if d == O.greedy_argmax(row):
                acc[j] = True
                if depth[j] > depth[best] or (last_tie and depth[j] == depth[best]):
                    best = j
        path, j = [], best
        while j != 0:
            path.append(j)
            j = int(node_parents[j - 1])
        path.reverse()
        return O.TreeResult([int(node_tokens[c - 1]) for c in path] + [O.greedy_argmax(target[best])],
                            path, len(path), status, n)
    return run


MUTATIONS = {
    "resample_from_p": ("residual_weights", lambda p, q: p.copy()),
    "residual_transposed": ("residual_weights", lambda p, q: np.maximum(q - p, 0.0)),
    "ratio_transposed": ("acceptance_ratio", lambda p, q: (q / p) if p > 0 else np.inf),
    "temperature_dropped": ("softmax_at_temperature",
                            lambda L, T: np.exp(L - L.max()) / np.exp(L - L.max()).sum()),
    "greedy_last_tie": ("greedy_argmax", _greedy_last_max),
    "inverse_cdf_ge": ("inverse_cdf", _icdf_ge),
    "row_shift": ("verify_sample_sequence", None),
    "stops_last_token_only": ("apply_stops", _stops_last_token_only),
    "stops_budget_ignored": ("apply_stops", lambda o, m, e, n=None: _apply_stops(o, m, e, None)),
    "tree_own_row": ("verify_tree_greedy_sequence", _tree_variant(own_row=True)),
    "tree_last_index_tie": ("verify_tree_greedy_sequence", _tree_variant(last_tie=True)),
    "top_p_full_mass": ("truncated_distribution", _trunc_variant(full_mass=True)),
    "top_k_drops_ties": ("truncated_distribution", _trunc_variant(strict_k=True)),
    "accept_margin_halved": ("accept_margin", lambda u, r: abs(u - r) / 2),
    "accept_margin_doubled": ("accept_margin", lambda u, r: abs(u - r) * 2),
    "accept_margin_of_clamped_ratio_minus_u": ("accept_margin", lambda u, r: min(1.0, r) - u),
    "inverse_cdf_margin_halved": ("inverse_cdf", _icdf_margin_scaled(0.5)),
    "inverse_cdf_margin_doubled": ("inverse_cdf", _icdf_margin_scaled(2.0)),
    "top_p_margin_halved": ("truncated_distribution", _top_p_margin_scaled(0.5)),
    "top_p_margin_doubled": ("truncated_distribution", _top_p_margin_scaled(2.0)),
    "bad_row_nan_unseen": ("row_has_distribution", lambda row: bool(np.isfinite(np.nanmax(row)))),
    "bad_row_all_neg_inf_unseen": ("row_has_distribution", lambda row: not np.isnan(np.max(row))),
}


def _pins_pass():
    checks = [pins.check_three_token_example, pins.check_greedy_tables,
              pins.check_expected_tokens, pins.check_inverse_cdf_convention,
              pins.check_greedy_tie_rule,
              lambda: pins.check_joint_law(3, 2, 0.7, 2),
              lambda: pins.check_joint_law(3, 1, 1.0, 1),
              pins.check_stops_match_step_by_step,
              pins.check_tree_figure, pins.check_tree_chain_equals_chain,
              pins.check_tree_matches_greedy_walk, pins.check_tree_ties_and_invalid_nodes,
              pins.check_truncation_against_counting, pins.check_top_k_one_is_greedy,
              lambda: pins.check_truncated_joint_law(4, 2, 0.8, 0, 0.7, 32),
              lambda: pins.check_accept_margin(cases=200, need_flips=40),
              lambda: pins.check_inverse_cdf_margin(cases=200, need_flips=60),
              lambda: pins.check_top_p_margin(cases=150, need_flips=40),
              pins.check_flagged_uses_every_margin,
              pins.check_rows_without_distribution, pins.check_truncated_entry_masks_nan]
    for c in checks:
        try:
            c()
        except (AssertionError, IndexError, ValueError, ZeroDivisionError, FloatingPointError):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    if fn is None:
        fn = _shifted_rows(O.verify_sample_sequence)
    monkeypatch.setattr(O, attr, fn)
    with np.errstate(all="ignore"):
        assert not _pins_pass(), f"mutation {name} went unnoticed"


def test_unmutated_oracle_passes():
    assert _pins_pass()
