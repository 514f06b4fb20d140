"""Pin checks for the float64 oracle, shared by the pin tests and the mutation tests.

Each function raises AssertionError when the oracle disagrees with something the
pages or plain mathematics fix.  The mutation tests plant plausible mistakes in
the oracle and require that at least one of these checks then fails.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np

from oracle import specverify_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def frac_list(xs):
    return [Fraction(x) for x in xs]


# ---------------------------------------------------------------------------------------
# Black-box integration of the oracle's step over its explicit uniforms.
#
# For fixed drafts the step is a function of (u_accept[0..g-1], u_sample).  Row i is kept
# iff u_accept[i] lies below a threshold t_i, and the sampled token is a non-decreasing step
# function of u_sample (ascending-id inverse CDF).  Thresholds and breakpoints are located
# by bisection on the oracle itself; the law of the emitted tokens is then the sum over the
# cells of the resulting product partition of [0,1)^(g+1), each evaluated at its centre.
# ---------------------------------------------------------------------------------------

_BISECT = 64


def _bisect(pred, lo=0.0, hi=1.0):
    """sup{u in [lo,hi] : pred(u)} for a predicate true on [lo, t) and false on [t, hi]."""
    if not pred(lo):
        return lo
    if pred(np.nextafter(hi, 0.0)):
        return hi
    for _ in range(_BISECT):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def step(P, Q, d, T, ua, us):
    g = len(d)
    return O.verify_sample_sequence(P, Q, np.asarray(d, dtype=np.int64), g, T,
                                    np.asarray(ua, dtype=np.float64), us)


def emitted_law(P, Q, d, T, step=step):
    """{tuple(emitted tokens): probability} of one step with drafts d, integrating over
    the uniforms by probing the oracle."""
    g = len(d)
    V = P.shape[1]
    thr = []
    for i in range(g):
        # make rows < i pass (u = 0) so that row i's decision is observable
        base = [0.0] * g

        def kept(u, i=i):
            ua = list(base)
            ua[i] = u
            return step(P, Q, d, T, ua, 0.5).m > i

        reachable = all(step(P, Q, d, T, [0.0] * g, 0.5).m > j for j in range(i))
        thr.append(_bisect(kept) if reachable else 0.5)
    law = {}
    for cell in itertools.product((0, 1), repeat=g):
        widths, centre = 1.0, []
        for i, side in enumerate(cell):
            lo, hi = (0.0, thr[i]) if side == 0 else (thr[i], 1.0)
            widths *= hi - lo
            centre.append(0.5 * (lo + hi))
        if widths <= 0.0:
            continue

        def last_tok(us):
            return step(P, Q, d, T, centre, us).tokens[-1]

        prev = 0.0
        for v in range(V):
            b = _bisect(lambda us: last_tok(us) <= v)
            if b > prev:
                toks = tuple(step(P, Q, d, T, centre, 0.5 * (prev + b)).tokens)
                assert toks[-1] == v
                law[toks] = law.get(toks, 0.0) + widths * (b - prev)
                prev = b
    return law


def softmax_T(logits, T):
    """Textbook temperature softmax, used only to state the target's own law."""
    z = np.asarray(logits, dtype=np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


# ---------------------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------------------

def check_three_token_example(tol=1e-12):
    """The worked example: kept mass (0.2,0.3,0.2), rejection 0.3, residual (1,0,0),
    output exactly p (M013 card §05; nxmr.cn 151309)."""
    G = golden("three_token_example.json")
    p = np.array([float(Fraction(x)) for x in G["p"]])
    q = np.array([float(Fraction(x)) for x in G["q"]])
    P = np.log(np.stack([p, p]))
    Q = np.log(q)[None, :]
    out = np.zeros(3)
    kept = np.zeros(3)
    for x in range(3):
        law = emitted_law(P, Q, [x], 1.0)
        for toks, pr in law.items():
            if len(toks) == 2:               # x kept (then a bonus token follows)
                kept[x] += q[x] * pr
                out[toks[0]] += q[x] * pr
            else:                            # rejected: the correction is the only token
                out[toks[0]] += q[x] * pr
    acc_prob = kept / q
    assert np.allclose(acc_prob, [float(Fraction(a)) for a in G["accept_prob"]], atol=tol, rtol=0), acc_prob
    assert np.allclose(kept, [float(Fraction(a)) for a in G["accepted_mass"]], atol=tol, rtol=0), kept
    assert abs((1 - kept.sum()) - float(Fraction(G["reject_mass"]))) < tol
    assert np.allclose(out, [float(Fraction(a)) for a in G["output"]], atol=tol, rtol=0), out
    # the residual branch alone: reject x = B and read the law of the correction
    res = np.zeros(3)
    law = emitted_law(P, Q, [1], 1.0)
    rej = sum(pr for t, pr in law.items() if len(t) == 1)
    for t, pr in law.items():
        if len(t) == 1:
            res[t[0]] += pr / rej
    assert np.allclose(res, [float(Fraction(a)) for a in G["residual"]], atol=tol, rtol=0), res
    return out


def check_greedy_tables():
    """Page tables: the draft is kept up to the first mismatch with the target's greedy
    choice, whose token replaces it (M013 card §03; tutorial §3.3)."""
    for case in golden("greedy_tables.json")["cases"]:
        vocab = sorted(set(case["draft"]) | set(case["target_greedy"]) | {"<other>"})
        ids = {w: i for i, w in enumerate(vocab)}
        V = len(vocab)
        k = len(case["draft"])
        rng = np.random.default_rng(7)
        rows = rng.normal(0, 1, size=(k + 1, V))
        for i, w in enumerate(case["target_greedy"]):
            rows[i, ids[w]] = 10.0
        d = np.array([ids[w] for w in case["draft"]])
        r = O.verify_greedy_sequence(rows, d, k)
        assert r.m == case["accepted"], (r.m, case)
        assert r.tokens == [ids[w] for w in case["committed"]], (r.tokens, case)
    # full agreement: k tokens plus the bonus argmax of row k (tutorial §5.3)
    rows = np.zeros((4, 6))
    for i, t in enumerate([3, 1, 4, 5]):
        rows[i, t] = 1.0
    r = O.verify_greedy_sequence(rows, np.array([3, 1, 4]), 3)
    assert r.m == 3 and r.tokens == [3, 1, 4, 5], r.tokens


def controlled_alpha_rows(alpha, gamma):
    """p = (a, 1-a, 0), q = (a, 0, 1-a): sum_v min(p, q) = a exactly.  Draft 0 is always kept
    (p = q), draft 2 always rejected (p = 0)."""
    with np.errstate(divide="ignore"):
        P = np.log(np.tile([alpha, 1 - alpha, 0.0], (gamma + 1, 1)))
        Q = np.log(np.tile([alpha, 0.0, 1 - alpha], (gamma, 1)))
    return P, Q


def expected_emitted_exact(alpha, gamma):
    """E[emitted per round] by exact enumeration of the draft patterns through the oracle,
    and the law of m."""
    P, Q = controlled_alpha_rows(alpha, gamma)
    E = 0.0
    pm = np.zeros(gamma + 1)
    for pat in itertools.product((0, 2), repeat=gamma):
        w = math.prod(alpha if x == 0 else 1 - alpha for x in pat)
        r = O.verify_sample_sequence(P, Q, np.array(pat), gamma, 1.0, np.full(gamma, 0.5), 0.5)
        E += w * len(r.tokens)
        pm[r.m] += w
    return E, pm


def check_expected_tokens():
    """Closed form (1 - a^(g+1))/(1 - a) and the values the pages print."""
    G = golden("expected_tokens.json")
    for row in G["printed"]:
        a, g = row["alpha"], row["gamma"]
        E, pm = expected_emitted_exact(a, g)
        assert abs(E - row["value"]) <= 0.5 * 10 ** (-row["printed_decimals"]) + 1e-12, (row, E)
        assert abs(E - (1 - a ** (g + 1)) / (1 - a)) < 1e-12
        # P(m = j) = a^j (1 - a) for j < g, a^g at g (tutorial §8)
        want = [a ** j * (1 - a) for j in range(g)] + [a ** g]
        assert np.allclose(pm, want, atol=1e-14), pm
        EM = sum(j * pm[j] for j in range(g + 1))
        assert abs(EM - a * (1 - a ** g) / (1 - a)) < 1e-12
    for row in G["misprinted"]:
        E, _ = expected_emitted_exact(row["alpha"], row["gamma"])
        assert abs(E - row["formula_on_same_page"]) < 1e-6, (row, E)


def random_tables(V, depth, seed, scale=1.5, zero_frac=0.0):
    """Conditional logits of a toy target and draft model: logits(prefix) per model."""
    rng = np.random.default_rng(seed)
    cache = {}

    def logits(model, prefix):
        key = (model, tuple(prefix))
        if key not in cache:
            x = rng.normal(0, scale, size=V)
            if zero_frac and model == "target":
                mask = rng.random(V) < zero_frac
                mask[rng.integers(V)] = False
                x[mask] = -np.inf
            cache[key] = x
        return cache[key]

    return logits


def check_joint_law(V, gamma, T, seed, zero_frac=0.0, tol=1e-9):
    """Brute force: draft tokens drawn autoregressively from the toy draft model, target rows
    aligned as in the tutorial's §4 table, the step's emitted prefix extended by the target's
    own sampling up to gamma+1 tokens must have exactly the target's autoregressive law
    (tutorial §7.3: every position keeps its conditional law)."""
    logits = random_tables(V, gamma + 1, seed, zero_frac=zero_frac)
    n = gamma + 1
    ext = {}
    for d in itertools.product(range(V), repeat=gamma):
        qd = 1.0
        for i in range(gamma):
            qd *= softmax_T(logits("draft", d[:i]), T)[d[i]]
        if qd == 0.0:
            continue
        P = np.stack([logits("target", d[:i]) for i in range(gamma + 1)])
        Q = np.stack([logits("draft", d[:i]) for i in range(gamma)])
        for toks, pr in emitted_law(P, Q, list(d), T).items():
            # extend with the target's own sampling up to n tokens
            frontier = {toks: qd * pr}
            while True:
                nxt = {}
                for seq, w in frontier.items():
                    if len(seq) == n:
                        ext[seq] = ext.get(seq, 0.0) + w
                        continue
                    pt = softmax_T(logits("target", seq), T)
                    for v in range(V):
                        if pt[v] > 0:
                            nxt[seq + (v,)] = nxt.get(seq + (v,), 0.0) + w * pt[v]
                if not nxt:
                    break
                frontier = nxt
    for seq in itertools.product(range(V), repeat=n):
        want = 1.0
        for j in range(n):
            want *= softmax_T(logits("target", seq[:j]), T)[seq[j]]
        got = ext.get(seq, 0.0)
        assert abs(got - want) < tol, (seq, got, want)


def check_inverse_cdf_convention():
    """Ascending ids, strict C_v > u*R: zero-weight ids are never returned."""
    w = np.array([0.0, 0.5, 0.0, 0.25, 0.25, 0.0])
    assert O.inverse_cdf(w, 0.0)[0] == 1
    assert O.inverse_cdf(w, 0.49999)[0] == 1
    assert O.inverse_cdf(w, 0.5)[0] == 3
    assert O.inverse_cdf(w, 0.75)[0] == 4
    assert O.inverse_cdf(w, np.nextafter(1.0, 0.0))[0] == 4
    assert O.inverse_cdf(w, 1.0)[0] == 4       # u outside [0,1): the last positive id


def check_greedy_tie_rule():
    row = np.array([1.0, 3.0, 2.0, 3.0, -np.inf, 3.0])
    assert O.greedy_argmax(row) == 1
    assert O.greedy_argmax(np.full(5, -np.inf)) == 0


# ------------------------------------------------------------------------------------------
# stops: speculative rounds with the oracle's verify and stops reproduce step-by-step decoding
# that ends at the first end token or at the length limit ([TUT] §12.3 asks exactly this of
# EOS, maximum length and the rejection position; §5.2 forbids anything after an EOS in the
# candidate block from reaching the cache)
# ------------------------------------------------------------------------------------------

def toy_model(seed, V, eos, eos_bias):
    """A deterministic toy language model: the logits after any prefix come from a generator
    seeded by (seed, prefix)."""
    def logits(prefix):
        x = np.random.default_rng([seed, len(prefix)] + [int(t) for t in prefix]).normal(0.0, 2.0, V)
        x[eos] += eos_bias
        return x
    return logits


def noisy_copy(model, seed, sigma):
    """A draft model: the target's logits plus seeded noise (high but imperfect agreement)."""
    def logits(prefix):
        x = model(prefix)
        return x + np.random.default_rng([seed, len(prefix)] + [int(t) for t in prefix]).normal(0.0, sigma, len(x))
    return logits


def ar_greedy_decode(target, prompt, eos, max_new):
    """Step-by-step greedy decoding: one target argmax per token (first index on ties), stop
    after the end token or after max_new tokens."""
    out = []
    while len(out) < max_new:
        t = int(np.argmax(target(prompt + out)))
        out.append(t)
        if t == eos:
            break
    return out


def spec_greedy_decode(target, draft, prompt, eos, max_new, gamma, max_rounds=200):
    """Speculative greedy decoding through the oracle: draft gamma tokens greedily, verify
    them against the target rows, cut the emit with apply_stops, append, repeat."""
    from oracle import specverify_oracle as O
    out = []
    for _ in range(max_rounds):
        prefix = prompt + out
        ds = []
        for _i in range(gamma):
            ds.append(int(np.argmax(draft(prefix + ds))))
        rows = np.stack([target(prefix + ds[:i]) for i in range(gamma + 1)])
        r = O.verify_greedy_sequence(rows, np.array(ds), gamma)
        toks = np.full((1, gamma + 1), -1, dtype=np.int64)
        toks[0, : len(r.tokens)] = r.tokens
        o2, _, st = O.apply_stops(toks, np.array([r.m]), eos, np.array([max_new - len(out)]))
        out += [int(t) for t in o2[0] if t >= 0]
        if st[0] & O.ST_STOPPED:
            return out
    raise AssertionError("speculative decoding did not stop")


def check_stops_match_step_by_step(cases=None):
    """Cases mix end tokens accepted inside a draft block, end tokens as the correction or
    bonus token, and budgets that cut a block (V = 10, id 0 the end token)."""
    cases = cases or [(seed, g, n, bias) for seed in range(10) for g in (1, 2, 4)
                      for n in (1, 3, 9, 25) for bias in (-1.0, 0.5)]
    for seed, gamma, max_new, bias in cases:
        V, eos = 10, 0
        target = toy_model(seed, V, eos, bias)
        draft = noisy_copy(target, seed + 100, 1.0)
        want = ar_greedy_decode(target, [3], eos, max_new)
        got = spec_greedy_decode(target, draft, [3], eos, max_new, gamma)
        assert got == want, (seed, gamma, max_new, bias, got, want)


# ---------------------------------------------------------------------------------------
# tree verification (tutorial §5.3): greedy acceptance along a draft tree
# ---------------------------------------------------------------------------------------

def check_tree_figure():
    """The tutorial's §5.3 tree, with three target continuations: the longer accepted
    branch wins, a branch stops at its first mismatch, and nothing is accepted when the
    first token already differs."""
    G = golden("tree_figure.json")
    names = G["nodes"]
    words = sorted(set(names) | {"<bonus>", "<other>", "root"})
    ids = {w: i for i, w in enumerate(words)}
    V = len(words)
    n = len(names)
    toks = np.array([ids[w] for w in names])
    par = np.array(G["parents"])
    for case in G["cases"]:
        rows = np.zeros((n + 1, V))
        for after, nxt in case["target_greedy_after"].items():
            r = 0 if after == "root" else names.index(after) + 1
            rows[r, ids[nxt]] = 1.0
        res = O.verify_tree_greedy_sequence(rows, toks, par, n)
        assert [names[j - 1] for j in res.path] == case["path"], (res, case)
        assert res.tokens == [ids[w] for w in case["emitted"]], (res, case)
        assert res.m == len(case["path"]) and res.status == 0


def check_tree_chain_equals_chain(cases=60, seed=5):
    """A chain tree (node j's parent is j-1) is the chain verification of the same drafts."""
    rng = np.random.default_rng(seed)
    for _ in range(cases):
        V = int(rng.integers(2, 9))
        n = int(rng.integers(0, 7))
        rows = rng.normal(0, 1, size=(n + 1, V)).round(1)
        am = [int(np.argmax(r)) for r in rows]
        d = np.array([am[i] if rng.random() < 0.7 else int(rng.integers(0, V)) for i in range(n)], dtype=np.int64)
        if n and rng.random() < 0.2:
            d[int(rng.integers(0, n))] = V + 3   # an id outside the row
        chain = O.verify_greedy_sequence(rows, d, n)
        tree = O.verify_tree_greedy_sequence(rows, d, np.arange(n), n)
        assert tree.tokens == chain.tokens and tree.m == chain.m and tree.status == chain.status, (tree, chain)
        assert tree.path == list(range(1, chain.m + 1))


def _greedy_walk(rows, toks, par, n):
    """The target's own greedy continuation, followed through the tree as long as the tree
    holds the next token as a child: a second statement of 'the longest accepted path' for
    trees whose siblings carry distinct tokens."""
    children = {}
    for j in range(1, n + 1):
        children.setdefault(int(par[j - 1]), {})[int(toks[j - 1])] = j
    node, path = 0, []
    while True:
        x = int(np.flatnonzero(rows[node] == rows[node].max())[0])
        nxt = children.get(node, {}).get(x)
        if nxt is None:
            return path, [int(toks[c - 1]) for c in path] + [x]
        path.append(nxt)
        node = nxt


def check_tree_matches_greedy_walk(cases=200, seed=11):
    rng = np.random.default_rng(seed)
    for _ in range(cases):
        V = int(rng.integers(3, 8))
        n = int(rng.integers(0, 12))
        par = np.array([int(rng.integers(0, j)) for j in range(1, n + 1)], dtype=np.int64)
        rows = rng.normal(0, 1, size=(n + 1, V)).round(1)
        toks = np.zeros(n, dtype=np.int64)
        used = {}
        for j in range(1, n + 1):
            p = int(par[j - 1])
            free = [v for v in range(V) if v not in used.get(p, set())]
            if not free:              # more children than ids: give the node up to the root
                par[j - 1] = 0
                p = 0
                free = [v for v in range(V) if v not in used.get(0, set())] or [0]
            am = int(np.flatnonzero(rows[p] == rows[p].max())[0])
            t = am if (am in free and rng.random() < 0.6) else int(rng.choice(free))
            toks[j - 1] = t
            used.setdefault(p, set()).add(t)
        if any(len(set(int(toks[c - 1]) for c in range(1, n + 1) if int(par[c - 1]) == p)) !=
               sum(1 for c in range(1, n + 1) if int(par[c - 1]) == p) for p in range(n + 1)):
            continue                  # duplicate siblings: the walk is not defined there
        res = O.verify_tree_greedy_sequence(rows, toks, par, n)
        path, emitted = _greedy_walk(rows, toks, par, n)
        assert res.path == path and res.tokens == emitted, (res, path, emitted)


def check_tree_ties_and_invalid_nodes():
    """Equal-depth accepted paths (two siblings with the same token): the lower node index
    wins.  A node whose parent index is not below its own is never accepted, nor is its
    subtree (bit 64); a candidate id outside [0, V) is a rejection (bit 1)."""
    V = 5
    rows = np.zeros((5, V))
    rows[0, 2] = 1.0      # root -> 2
    rows[1, 3] = 1.0      # after node 1 -> 3
    rows[2, 3] = 1.0      # after node 2 -> 3
    rows[3, 4] = 1.0
    rows[4, 1] = 1.0
    # nodes: 1 = 2 (root), 2 = 2 (root), 3 = 3 (under 2), 4 = 3 (under 1)
    res = O.verify_tree_greedy_sequence(rows, np.array([2, 2, 3, 3]), np.array([0, 0, 2, 1]), 4)
    assert res.path == [2, 3] and res.tokens == [2, 3, 4] and res.status == 0, res
    res = O.verify_tree_greedy_sequence(rows, np.array([2, 2, 3, 3]), np.array([0, 0, 1, 1]), 4)
    assert res.path == [1, 3], res
    # node 2 names itself as its parent; node 3 hangs below it
    res = O.verify_tree_greedy_sequence(rows, np.array([7, 2, 3]), np.array([0, 2, 2]), 3)
    assert res.status == O.ST_BAD_TREE | O.ST_BAD_DRAFT and res.path == [] and res.tokens == [2], res


# ---------------------------------------------------------------------------------------
# truncated sampling (NXM / KB §10: truncation must show in p and q): top-k, then top-p
# ---------------------------------------------------------------------------------------

def kept_by_counting(logits, T, top_k, top_p):
    """The kept set stated element by element: v survives top-k iff fewer than k logits are
    strictly larger; it survives top-p iff the top-k-kept mass strictly above its logit is
    below top_p times the whole top-k-kept mass (it is needed to reach the target)."""
    x = np.asarray(logits, dtype=np.float64)
    V = len(x)
    p = softmax_T(x, T)
    keep = np.ones(V, dtype=bool)
    if 0 < top_k < V:
        keep = np.array([np.sum(x > x[v]) < top_k for v in range(V)])
    if 0.0 < top_p < 1.0:
        mass_k = np.sum(p[keep])
        keep = keep & np.array([np.sum(p[keep & (x > x[v])]) < top_p * mass_k for v in range(V)])
    return keep


def check_truncation_against_counting(cases=300, seed=21):
    rng = np.random.default_rng(seed)
    for c in range(cases):
        V = int(rng.integers(1, 40))
        x = rng.normal(0, 2, size=V)
        if c % 3 == 0:
            x = np.round(x * 2) / 2            # many exact ties, as bf16 logits have
        T = float(rng.choice([0.5, 1.0, 1.7]))
        k = int(rng.choice([0, 1, 2, 5, V, V + 3, -1]))
        tp = float(rng.choice([1.0, 0.0, 0.3, 0.75, 0.95, 0.999, 1.5]))
        want = kept_by_counting(x, T, k, tp)
        got, _ = O.truncated_distribution(x, T, k, tp)
        assert np.array_equal(got > 0, want), (x, T, k, tp, got, want)
        p = softmax_T(x, T)
        assert np.allclose(got[want], p[want] / p[want].sum(), rtol=1e-12, atol=0)


def check_top_k_one_is_greedy(cases=200, seed=22):
    """top_k = 1 leaves one id on each side, so sampling verification with drafts from q'
    (its argmax) is greedy verification, for any uniforms."""
    rng = np.random.default_rng(seed)
    for _ in range(cases):
        V, g = int(rng.integers(2, 30)), int(rng.integers(0, 6))
        P = rng.normal(0, 2, size=(g + 1, V))
        Q = P[:g] + rng.normal(0, 1.0, size=(g, V))
        d = np.argmax(Q, axis=1) if g else np.zeros(0, dtype=np.int64)
        ua, us = rng.random(g), float(rng.random())
        s1 = O.verify_sample_sequence(P, Q, d, g, float(rng.choice([0.6, 1.0])), ua, us, top_k=1)
        s0 = O.verify_greedy_sequence(P, d, g)
        assert s1.tokens == s0.tokens and s1.m == s0.m, (s1, s0)


def check_truncation_off_switches(seed=23):
    rng = np.random.default_rng(seed)
    V, g = 17, 3
    P = rng.normal(0, 2, size=(g + 1, V))
    Q = P[:g] + rng.normal(0, 1.0, size=(g, V))
    d = rng.integers(0, V, size=g)
    ua, us = rng.random(g), 0.37
    base = O.verify_sample_sequence(P, Q, d, g, 0.9, ua, us)
    for k, tp in [(0, 1.0), (-3, 1.0), (V, 1.0), (V + 1, 2.0), (0, 0.0), (0, -0.5)]:
        r = O.verify_sample_sequence(P, Q, d, g, 0.9, ua, us, top_k=k, top_p=tp)
        assert r.tokens == base.tokens and r.m == base.m and r.p_draft == base.p_draft, (k, tp)


def check_truncated_joint_law(V, gamma, T, top_k, top_p, seed, tol=1e-9):
    """Brute force with truncation on both sides: drafts drawn from the draft's truncated
    distribution, the step's emitted prefix extended by the target's truncated sampling,
    gives exactly the truncated target's autoregressive law."""
    logits = random_tables(V, gamma + 1, seed)

    def tr(x):
        keep = kept_by_counting(x, T, top_k, top_p)
        p = softmax_T(x, T) * keep
        return p / p.sum()

    def tstep(P, Q, d, T_, ua, us):
        return O.verify_sample_sequence(P, Q, np.asarray(d, dtype=np.int64), len(d), T_,
                                        np.asarray(ua, dtype=np.float64), us, top_k=top_k, top_p=top_p)

    n = gamma + 1
    ext = {}
    for d in itertools.product(range(V), repeat=gamma):
        qd = 1.0
        for i in range(gamma):
            qd *= tr(logits("draft", d[:i]))[d[i]]
        if qd == 0.0:
            continue
        P = np.stack([logits("target", d[:i]) for i in range(gamma + 1)])
        Q = np.stack([logits("draft", d[:i]) for i in range(gamma)])
        for toks, pr in emitted_law(P, Q, list(d), T, step=tstep).items():
            frontier = {toks: qd * pr}
            while True:
                nxt = {}
                for sq, w in frontier.items():
                    if len(sq) == n:
                        ext[sq] = ext.get(sq, 0.0) + w
                        continue
                    pt = tr(logits("target", sq))
                    for v in range(V):
                        if pt[v] > 0:
                            nxt[sq + (v,)] = nxt.get(sq + (v,), 0.0) + w * pt[v]
                if not nxt:
                    break
                frontier = nxt
    for sq in itertools.product(range(V), repeat=n):
        want = 1.0
        for j in range(n):
            want *= tr(logits("target", sq[:j]))[sq[j]]
        assert abs(ext.get(sq, 0.0) - want) < tol, (sq, ext.get(sq, 0.0), want)


# ---------------------------------------------------------------------------------------
# decision margins: every margin the oracle reports is the distance from its uniform (or
# mass target) to the point where the decision it flags actually changes.  Parity tests
# exempt sequences whose margin is below 1e-5 from the bit-exact check (the near-tied
# decisions [TUT] §12.3 tells apart from real mismatches), so a margin computed too large
# would hide a real mismatch and one computed too small would widen the exemption.
# ---------------------------------------------------------------------------------------

_IN, _OUT = 1.0 - 1e-6, 1.0 + 1e-6


def _one_row_case(rng, V):
    T = float(rng.choice([0.6, 1.0, 1.4]))
    P = rng.normal(0, 1.5, size=(2, V))
    Q = P[:1] + rng.normal(0, float(rng.choice([0.1, 0.5, 1.5])), size=(1, V))
    d = np.array([int(rng.integers(0, V))])
    return P, Q, d, T


def check_accept_margin(cases=400, seed=31, need_flips=100):
    """Moving u_accept toward p(d)/q(d) by the reported margin times (1 - 1e-6) keeps the
    decision; by (1 + 1e-6) it flips it (where the moved u stays in [0, 1))."""
    rng = np.random.default_rng(seed)
    flips = 0
    for _ in range(cases):
        P, Q, d, T = _one_row_case(rng, int(rng.integers(2, 12)))
        u = float(rng.random())
        res = O.verify_sample_sequence(P, Q, d, 1, T, np.array([u]), 0.5)
        kept = res.m == 1
        a = res.accept_margins[0]
        assert a >= 0.0
        s = 1.0 if kept else -1.0             # kept: u < r, so r lies above u

        def keeps(v):
            return O.verify_sample_sequence(P, Q, d, 1, T, np.array([v]), 0.5).m == 1
        if a < 1e-9:
            continue
        u_in, u_out = u + s * a * _IN, u + s * a * _OUT
        if 0.0 <= u_in < 1.0:
            assert keeps(u_in) == kept, (u, a, u_in, kept)
        if 0.0 <= u_out < 1.0:
            assert keeps(u_out) != kept, (u, a, u_out, kept)
            flips += 1
        elif kept:
            # r >= 1: every u in [u, 1) keeps the draft
            for v in (u, 0.5 * (u + 1.0), float(np.nextafter(1.0, 0.0))):
                assert keeps(v)
    assert flips >= need_flips, flips


def check_inverse_cdf_margin(cases=400, seed=32, need_flips=150):
    """Moving u by the reported inverse-CDF margin times (1 - 1e-6), either way, keeps the
    token; by (1 + 1e-6) toward the nearer cell edge it changes it.  Checked on the function
    itself and on the draw of a whole step (correction or bonus)."""
    rng = np.random.default_rng(seed)
    flips = 0
    for c in range(cases):
        V = int(rng.integers(1, 16))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if not w.any():
            w[int(rng.integers(0, V))] = 1.0
        u = float(rng.random())
        v, a, _ = O.inverse_cdf(w, u)
        assert a >= 0.0
        if a < 1e-9:
            continue
        for s in (-1.0, 1.0):
            ui = u + s * a * _IN
            if 0.0 <= ui < 1.0:
                assert O.inverse_cdf(w, ui)[0] == v, (w, u, a, ui)
        # the nearer cell edge is crossed on one side; when a moved u leaves [0, 1) that edge
        # may be the end of the range itself, so only cases with both inside are required
        outs = [u + s * a * _OUT for s in (-1.0, 1.0)]
        if all(0.0 <= x < 1.0 for x in outs):
            assert any(O.inverse_cdf(w, x)[0] != v for x in outs), (w, u, a)
            flips += 1
    assert flips >= need_flips, flips
    # the same on whole steps: the sample margin is the margin of the draw actually made
    step_flips = 0
    for c in range(cases // 2):
        P, Q, d, T = _one_row_case(rng, int(rng.integers(2, 10)))
        ua = np.array([float(rng.random())])
        us = float(rng.random())
        res = O.verify_sample_sequence(P, Q, d, 1, T, ua, us)
        a = res.sample_margin
        if not (1e-9 <= a < 1.0):
            continue

        def tok(x):
            r = O.verify_sample_sequence(P, Q, d, 1, T, ua, x)
            assert r.m == res.m
            return r.tokens[-1]
        for s in (-1.0, 1.0):
            x = us + s * a * _IN
            if 0.0 <= x < 1.0:
                assert tok(x) == res.tokens[-1]
        outs = [us - a * _OUT, us + a * _OUT]
        if all(0.0 <= x < 1.0 for x in outs):
            assert any(tok(x) != res.tokens[-1] for x in outs)
            step_flips += 1
    assert step_flips >= need_flips // 3, step_flips


def check_top_p_margin(cases=300, seed=33, need_flips=100):
    """Moving top_p by the reported crossing margin times (1 - 1e-6), either way, keeps the
    kept set; by (1 + 1e-6) toward the nearer crossing it changes it."""
    rng = np.random.default_rng(seed)
    flips = 0
    for c in range(cases):
        V = int(rng.integers(2, 30))
        x = rng.normal(0, 2, size=V)
        if c % 3 == 0:
            x = np.round(x * 2) / 2
        T = float(rng.choice([0.5, 1.0, 1.7]))
        k = int(rng.choice([0, 3, 8]))
        tp = float(rng.uniform(0.05, 0.95))
        dist, a = O.truncated_distribution(x, T, k, tp)
        assert a >= 0.0
        kept = dist > 0
        if a < 1e-9 or not math.isfinite(a):
            continue
        for s in (-1.0, 1.0):
            t = tp + s * a * _IN
            if 0.0 < t < 1.0:
                assert np.array_equal(O.truncated_distribution(x, T, k, t)[0] > 0, kept), (x, tp, a, t)
        outs = [tp - a * _OUT, tp + a * _OUT]
        if all(0.0 < t < 1.0 for t in outs):
            assert any(not np.array_equal(O.truncated_distribution(x, T, k, t)[0] > 0, kept) for t in outs)
            flips += 1
    assert flips >= need_flips, flips
    # off: no crossing, no margin
    assert O.truncated_distribution(np.array([0.0, 1.0]), 1.0, 0, 1.0)[1] == math.inf


def check_flagged_uses_every_margin():
    """flagged() looks at every acceptance margin of the step and at its draw's margin."""
    r = O.SequenceResult([1], 0, 0, 2, False, [0.1, 0.1], [0.1, 0.1], 0.5, [0.5, 2e-6], 0.3)
    assert r.flagged(1e-5) and not r.flagged(1e-6)
    r.accept_margins = [0.5, 0.5]
    r.sample_margin = 5e-6
    assert r.flagged(1e-5) and not r.flagged(1e-6)


def check_rows_without_distribution():
    """A row the sampling step reads whose max is not finite, or which holds a NaN, defines no
    softmax (exp(L/T - max L/T) is 0/0 or NaN): the sequence carries ST_BAD_ROW.  Rows it does
    not read (past num_draft) and greedy sequences are not marked; ordinary rows never are."""
    rng = np.random.default_rng(5)
    V, g = 40, 3
    base_t = rng.normal(0, 2, (g + 1, V))
    base_q = base_t[:g] + rng.normal(0, 0.5, (g, V))
    drafts = np.array([3, 7, 11])
    u = np.array([0.3, 0.6, 0.9])

    def status(t, q, gamma=g, T=1.0):
        return O.verify_sample_sequence(t, q, drafts, gamma, T, u, 0.5).status

    assert status(base_t, base_q) & O.ST_BAD_ROW == 0
    for name, put in [("all -inf target", lambda t, q: t.__setitem__(1, -np.inf)),
                      ("all -inf draft", lambda t, q: q.__setitem__(0, -np.inf)),
                      ("all -inf bonus row", lambda t, q: t.__setitem__(g, -np.inf)),
                      ("NaN logit", lambda t, q: t.__setitem__((2, 5), np.nan)),
                      ("+inf logit", lambda t, q: q.__setitem__((1, 9), np.inf))]:
        t, q = base_t.copy(), base_q.copy()
        put(t, q)
        st = status(t, q)
        assert st & O.ST_BAD_ROW, name
        # the same rows under truncation: marked, and the oracle does not fail on them
        assert O.verify_sample_sequence(t, q, drafts, g, 1.0, u, 0.5, top_k=5, top_p=0.9).status & O.ST_BAD_ROW
    # a row past num_draft is not read
    t = base_t.copy()
    t[3] = -np.inf
    assert status(t, base_q, gamma=2) & O.ST_BAD_ROW == 0
    # a greedy sequence's rows with -inf logits keep their argmax (lowest id on ties)
    t = base_t.copy()
    t[1] = -np.inf
    r = O.verify_greedy_sequence(t, drafts, g)
    assert r.status & O.ST_BAD_ROW == 0
    # masked ids (some -inf, a finite max) are ordinary
    t = base_t.copy()
    t[:, ::2] = -np.inf
    assert status(t, base_q) & O.ST_BAD_ROW == 0


def check_truncated_entry_masks_nan():
    """The truncated entry point's reading: a NaN logit is an id that is never kept, so a row
    with a NaN and a finite max is ordinary there and its result equals that of the same row with
    the NaN replaced by -inf; a row of NaN and -inf only has no finite max and is marked."""
    rng = np.random.default_rng(6)
    V, g = 30, 2
    t = rng.normal(0, 2, (g + 1, V))
    q = t[:g] + rng.normal(0, 0.5, (g, V))
    drafts = np.array([4, 9])
    u = np.array([0.2, 0.7])
    tn = t.copy()
    tn[1, 6] = np.nan
    ti = t.copy()
    ti[1, 6] = -np.inf
    for k, p in [(0, 1.0), (5, 1.0), (0, 0.8), (6, 0.9)]:
        a = O.verify_sample_sequence(tn, q, drafts, g, 1.0, u, 0.4, k, p, nan_masked=True)
        b = O.verify_sample_sequence(ti, q, drafts, g, 1.0, u, 0.4, k, p)
        assert a.status & O.ST_BAD_ROW == 0
        assert (a.tokens, a.m, a.status) == (b.tokens, b.m, b.status)
    # without the masking the NaN row has no distribution
    assert O.verify_sample_sequence(tn, q, drafts, g, 1.0, u, 0.4).status & O.ST_BAD_ROW
    qn = q.copy()
    qn[0] = np.nan
    qn[0, 2] = -np.inf
    assert O.verify_sample_sequence(t, qn, drafts, g, 1.0, u, 0.4, 5, 0.9, nan_masked=True).status & O.ST_BAD_ROW
