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
}


def _pins_pass():
    checks = [pins.check_three_token_example, pins.check_greedy_tables,
              pins.check_expected_tokens, pins.check_inverse_cdf_convention,
              pins.check_greedy_tie_rule,
              lambda: pins.check_joint_law(3, 2, 0.7, 2),
              lambda: pins.check_joint_law(3, 1, 1.0, 1),
              pins.check_stops_match_step_by_step]
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
