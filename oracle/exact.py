"""Exact-fraction law of one verification step on a tiny vocabulary.

TEST INFRASTRUCTURE (same rules as specverify_oracle.py: tests/, smoke() and the
bench's CPU baseline only).

The three-token worked example of the "M013" knowledge-base card, §05, and of
nxmr.cn news 151309 is checked there by enumerating probability mass in exact
fractions instead of by random frequencies.  This module does the same
enumeration for any small p, q given as Fractions: the draft x is drawn from q;
it is kept with probability min(1, p(x)/q(x)); otherwise the replacement is drawn
from the residual max(p - q, 0) normalised by its total R.  The result is the
law of the emitted token together with the intermediate masses the pages print.

`residual="p"` plants the wrong variant the card warns about (re-sampling from p
after a rejection) so that tests can show the pins catch it.
"""
from __future__ import annotations

from fractions import Fraction
from typing import Dict, List, Sequence


def one_step_law(p: Sequence[Fraction], q: Sequence[Fraction], residual: str = "max") -> Dict[str, object]:
    V = len(p)
    assert len(q) == V and sum(p) == 1 and sum(q) == 1
    accept_prob: List[Fraction] = []
    accepted: List[Fraction] = []
    for x in range(V):
        if q[x] == 0:
            a = Fraction(1) if p[x] > 0 else Fraction(0)
        else:
            a = min(Fraction(1), p[x] / q[x])
        accept_prob.append(a)
        accepted.append(q[x] * a)          # mass of "x drafted and kept"
    reject = 1 - sum(accepted)
    if residual == "max":
        w = [max(p[x] - q[x], Fraction(0)) for x in range(V)]
    elif residual == "p":
        w = list(p)
    else:
        raise ValueError(residual)
    total = sum(w)
    r = [x / total for x in w] if total != 0 else [Fraction(0)] * V
    output = [accepted[x] + reject * r[x] for x in range(V)]
    return {"accept_prob": accept_prob, "accepted": accepted, "reject": reject,
            "residual_unnormalised": w, "residual": r, "output": output}
