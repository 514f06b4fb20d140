"""Float64 CPU oracle for the batched speculative-decoding verify-and-commit step.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg may import or run this module.  The product path (the CUDA library
and its Python binding) never imports it and shares no code with it.

It is a plain, slow, deliberately unoptimised restatement of what the step
computes, one sequence at a time, in float64 (bf16 and fp32 inputs widen to
float64 exactly).  Sources, by page title and section:

  [KB]  "M013" card of the ai-infra knowledge base (xuujii.github.io), §02-§06:
        greedy table (§03), acceptance min(1,p/q) with p, q the real sampling
        distributions after temperature (§04), the three-token worked example and
        the residual max(p-q,0)/R with the R = 0 remark (§05), commit and KV
        rollback pseudocode (§06).
  [TUT] "投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡" (richardf123.github.io),
        §2 (contiguous prefix), §3 (greedy), §4 (logit alignment), §5.2-§5.3 (trim
        to t+m, then t+m+1; bonus), §7.1-§7.3 (acceptance, residual, multi-token).
  [APP] "学徒的草稿：推测解码与大模型的加速哲学" (carrie-l.github.io), part 2,
        Steps 3-4 (accept when p >= q, else with probability p/q; residual; bonus).
  [NXM] nxmr.cn news 151309: the same three-token example, exact-fraction check,
        "R = 0 must not produce NaN", temperature/top-p must be reflected in p and q.

Readings where the pages leave a step open:
  * Rows arrive pre-aligned: target row i judges draft i, row 0 is the saved
    boundary prediction, row gamma_b is the bonus row ([TUT] §4 table).
  * Acceptance is the strict test u < min(1, r) with r = p(d)/q(d); when q(d) = 0,
    r = +inf if p(d) > 0, and r = 0 whenever p(d) = 0.
  * Greedy ties resolve to the lowest token id ([KB] §03 asks for a fixed rule).
  * Inverse CDF in ascending id order: the token is the smallest v with
    C_v > u * C_{V-1}, C the running sum of the weights; if none qualifies
    (only possible when u >= 1) the last id with positive weight is taken.
  * A rejection whose residual mass R is exactly 0 (unreachable in exact maths,
    [KB] §05, [NXM]) samples from p_m instead and sets status bit 2.
  * A draft id outside [0, V) is a rejection at that row (status bit 1); a
    num_draft outside [0, gmax] is clamped (status bit 4).
  * Temperature T <= 0 (or NaN) marks a greedy sequence; otherwise p = softmax(P/T)
    and q = softmax(Q/T), the same T on both sides.
  * Truncated sampling ([NXM] and [KB] §10: temperature, top-p or any other logits processing
    that changes the distribution must show in p and q; [TUT] §7's pseudocode leaves top-p
    out).  The same truncation is applied to both sides, each to its own distribution at T:
    top-k keeps the ids whose logit is at least the k-th largest logit (ties kept; k <= 0 or
    k >= V: off); top-p then keeps, of those, the ids whose logit is at least the largest
    value t with mass(logit >= t) >= top_p * mass(kept by top-k) (ties kept; top_p outside
    (0, 1): off); the kept probabilities are renormalised.  Acceptance, residual and the
    bonus draw then use these p' and q'.
  * Tree verification ([TUT] §5.3: the target checks every node of a draft tree in one
    forward and keeps the longest accepted root-to-leaf path; [KB] §01, §06: a tree has its
    own rules, and its branches need their own cache bookkeeping).  The pages give no
    sampling rule for trees, so trees are verified greedily: node j is accepted iff its
    parent is and its token equals the argmax of the parent's target row; the deepest
    accepted node (the lowest index among equal depths) ends the path; the emitted tokens
    are the path's, then the argmax of its last node's row.  A node whose parent index is
    not smaller than its own is never accepted (status bit 64).
  * Stops ([TUT] §5.2 "common mistakes": nothing after an EOS in the candidate block
    may reach the cache; §12.3: EOS, maximum length and the rejection position must
    agree with step-by-step decoding; [KB] §03: an end token or a length limit may end
    the round early).  A round's emit d_0..d_{m-1}, tok is cut after its first EOS and
    to the sequence's remaining token budget; the last emitted token is, as a
    correction token is, not yet fed to the models, so m becomes (tokens emitted) - 1.

Parity pins: see tests/test_oracle_pins.py.  Every function below is pinned by at
least one test against values the pages print, closed forms, or brute force.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

# status bits reported per sequence
ST_BAD_DRAFT = 1
ST_R_ZERO = 2
ST_CLAMPED_GAMMA = 4
ST_HISTORY_FULL = 8
ST_STOPPED = 32
ST_BAD_TREE = 64
ST_BAD_ROW = 128


def widen(row: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bit patterns (uint16) or float32 -> float64, exactly."""
    if dtype == "bf16":
        return (row.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(row, dtype=np.float32).astype(np.float64)


def softmax_at_temperature(logits: np.ndarray, T: float) -> np.ndarray:
    """p_v = exp(L_v/T - max_u L_u/T) / sum_w exp(L_w/T - max_u L_u/T).

    [KB] §04 and [NXM]: p and q are the distributions actually sampled from, after
    temperature; the same T divides both sides.
    """
    z = logits / T
    z = z - np.max(z)
    e = np.exp(z)
    return e / np.sum(e)


def row_has_distribution(row: np.ndarray) -> bool:
    """softmax(L/T) is defined on a row iff its max is finite and no logit is NaN: otherwise
    exp(L/T - max L/T) is 0/0 (every logit -inf), NaN (a +inf) or NaN-poisoned (np.max returns
    NaN when any logit is NaN)."""
    return bool(np.isfinite(np.max(row)))


def truncated_distribution(logits: np.ndarray, T: float, top_k: int = 0, top_p: float = 1.0):
    """p' = softmax(L/T) restricted to the ids top-k and then top-p keep, renormalised.

    top-k (0 < k < V) keeps the ids whose logit is >= the k-th largest logit (ties kept).
    top-p (0 < top_p < 1) keeps, of those, the ids whose logit is >= t*, the largest logit
    value t among them with sum(p over kept ids with logit >= t) >= top_p * sum(p over kept
    ids) (ties at t* kept).  Returns (p', margin): margin is how far the top-p crossing sits
    from its target, |cum(t*) - target| and |cum(next value above t*) - target|, relative to
    the kept mass (inf when top-p is off), used only to flag near-ties in parity tests.
    """
    p = softmax_at_temperature(logits, T)
    V = len(logits)
    keep = np.ones(V, dtype=bool)
    if 0 < top_k < V:
        tau_k = np.sort(logits)[::-1][top_k - 1]
        keep &= logits >= tau_k
    margin = math.inf
    if 0.0 < top_p < 1.0:
        vals, inv = np.unique(logits[keep], return_inverse=True)     # ascending distinct values
        mass = np.bincount(inv, weights=p[keep], minlength=len(vals))
        cum = np.cumsum(mass[::-1])                                   # from the largest value down
        total = float(cum[-1])
        target = top_p * total
        j = int(np.flatnonzero(cum >= target)[0])
        tau_p = vals[::-1][j]
        keep &= logits >= tau_p
        above = float(cum[j - 1]) if j > 0 else 0.0
        margin = min(float(cum[j]) - target, target - above) / total
    w = np.where(keep, p, 0.0)
    return w / np.sum(w), margin


def greedy_argmax(logits: np.ndarray) -> int:
    """g = argmax_v L_v, the lowest id among equal maxima ([TUT] §3, [KB] §03)."""
    best = np.max(logits)
    return int(np.flatnonzero(logits == best)[0])


def acceptance_ratio(p_d: float, q_d: float) -> float:
    """r = p(d)/q(d), with q(d) = 0 read as +inf when p(d) > 0 and 0 when p(d) = 0."""
    if p_d == 0.0:
        return 0.0
    if q_d == 0.0:
        return math.inf
    return p_d / q_d


def accept_draft(p_d: float, q_d: float, u: float) -> bool:
    """Accept draft d iff u < min(1, p(d)/q(d)) ([TUT] §7.1; [APP] Step 3: a draft
    with p >= q is always kept, otherwise kept with probability p/q)."""
    return u < min(1.0, acceptance_ratio(p_d, q_d))


def accept_margin(u: float, r: float) -> float:
    """|u - r|: how far the uniform of an acceptance test sits from the ratio it is compared
    with.  The decision u < min(1, r) can only change where u crosses r (for r >= 1, u in
    [0, 1) never does), so this is the distance to the decision boundary, used only to flag
    near-ties in parity tests (a fp32 evaluation of p and q may put r on the other side)."""
    return abs(u - r)


def residual_weights(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """w_v = max(p_v - q_v, 0); R = sum_v w_v = 1 - sum_v min(p_v, q_v) ([TUT] §7.2)."""
    return np.maximum(p - q, 0.0)


def inverse_cdf(weights: np.ndarray, u: float):
    """Sample an id from weights/sum(weights) with the explicit uniform u.

    C_v = sum_{k<=v} w_k in ascending id order; the token is the smallest v with
    C_v > u * C_{V-1}.  Returns (token, margin, total) where margin =
    min(u - C_{v-1}/C_{V-1}, C_v/C_{V-1} - u) is how far u sits from the nearest
    decision boundary (used only to flag near-ties in parity tests).
    """
    C = np.cumsum(weights)
    total = float(C[-1])
    target = u * total
    hits = np.flatnonzero(C > target)
    if hits.size:
        v = int(hits[0])
    else:
        v = int(np.flatnonzero(weights > 0)[-1])
    lo = float(C[v - 1]) if v > 0 else 0.0
    hi = float(C[v])
    margin = min(u - lo / total, hi / total - u) if total > 0 else 0.0
    return v, margin, total


@dataclasses.dataclass
class SequenceResult:
    tokens: List[int]               # the m+1 emitted tokens: d_0..d_{m-1}, then correction/bonus
    m: int                          # accepted drafts
    status: int
    gamma: int                      # num_draft after clamping
    greedy: bool
    p_draft: List[float]            # p_i(d_i) for i < gamma (sampling), NaN where undefined
    q_draft: List[float]
    mass: float                     # mass the last token was drawn from (R, or sum p on bonus)
    accept_margins: List[float]     # |u_i - r_i| for the decisions actually taken (i <= m)
    sample_margin: float            # inverse-CDF margin (inf for greedy)

    def flagged(self, tol: float = 1e-5) -> bool:
        return any(a < tol for a in self.accept_margins) or self.sample_margin < tol


def verify_greedy_sequence(target: np.ndarray, drafts: np.ndarray, gamma: int) -> SequenceResult:
    """Greedy verification of one sequence ([TUT] §3.3, §4, §5.3; [KB] §03).

    target: float64 [>= gamma+1, V] aligned rows.  m is the first i < gamma with
    d_i != argmax(row i), else gamma; the emitted token is argmax(row m), which is the
    target's replacement on a mismatch and the bonus token on full acceptance.
    """
    V = target.shape[1]
    status = 0
    m = gamma
    for i in range(gamma):
        d = int(drafts[i])
        if not (0 <= d < V):
            status |= ST_BAD_DRAFT
        if d != greedy_argmax(target[i]):
            m = i
            break
    tok = greedy_argmax(target[m])
    toks = [int(x) for x in drafts[:m]] + [tok]
    nan = [math.nan] * gamma
    return SequenceResult(toks, m, status, gamma, True, nan, list(nan), math.nan, [], math.inf)


def verify_sample_sequence(target: np.ndarray, draft: np.ndarray, drafts: np.ndarray,
                           gamma: int, T: float, u_accept: np.ndarray, u_sample: float,
                           top_k: int = 0, top_p: float = 1.0, nan_masked: bool = False) -> SequenceResult:
    """Sampling verification of one sequence ([TUT] §7.1-§7.3; [APP] Steps 3-4; [KB] §05-§06).

    For i = 0..gamma-1, left to right: p_i = softmax(P_i/T), q_i = softmax(Q_i/T),
    accept d_i iff u_accept[i] < min(1, p_i(d_i)/q_i(d_i)); stop at the first rejection
    m.  On a rejection the correction is drawn from max(p_m - q_m, 0)/R with u_sample; on
    full acceptance the bonus token is drawn from p_gamma with u_sample.  With top_k / top_p
    set, p and q are the truncated distributions (truncated_distribution) on both sides.
    nan_masked: a NaN logit is read as -inf (an id that is never kept), the reading of the
    truncated entry point, whose exact key search counts no NaN key.
    """
    V = target.shape[1]
    status = 0
    if nan_masked:
        target = np.where(np.isnan(target), -np.inf, target)
        draft = np.where(np.isnan(draft), -np.inf, draft)
    # A row whose maximum is not finite, or which holds a NaN (every logit -inf, a +inf or a
    # NaN), has no softmax: exp(L/T - max L/T) is NaN or 0/0.  The sequence is marked
    # ST_BAD_ROW when any row it reads (target rows 0..gamma, draft rows 0..gamma-1) is such
    # a row; what follows is then not a defined result, and parity tests check the mark and
    # that the step is well formed.
    for row in list(target[: gamma + 1]) + list(draft[:gamma]):
        if not row_has_distribution(row):
            status |= ST_BAD_ROW
    if status & ST_BAD_ROW:
        nan = [math.nan] * gamma
        return SequenceResult([0], 0, status, gamma, False, nan, list(nan), math.nan, [], math.inf)
    m = gamma
    p_d: List[float] = []
    q_d: List[float] = []
    margins: List[float] = []
    p_m = q_m = None
    truncated = (0 < top_k < V) or (0.0 < top_p < 1.0)

    def dist(row):
        if not truncated:
            return softmax_at_temperature(row, T)
        d, tm = truncated_distribution(row, T, top_k, top_p)
        margins.append(tm)
        return d

    for i in range(gamma):
        p = dist(target[i])
        q = dist(draft[i])
        d = int(drafts[i])
        if 0 <= d < V:
            pd, qd = float(p[d]), float(q[d])
            p_d.append(pd)
            q_d.append(qd)
            margins.append(accept_margin(float(u_accept[i]), acceptance_ratio(pd, qd)))
            ok = accept_draft(pd, qd, float(u_accept[i]))
        else:
            status |= ST_BAD_DRAFT
            p_d.append(math.nan)
            q_d.append(math.nan)
            ok = False
        if not ok:
            m = i
            p_m, q_m = p, q
            break
    p_d += [math.nan] * (gamma - len(p_d))
    q_d += [math.nan] * (gamma - len(q_d))
    if m < gamma:
        w = residual_weights(p_m, q_m)
        if np.sum(w) > 0.0:
            tok, smargin, mass = inverse_cdf(w, float(u_sample))
        else:
            status |= ST_R_ZERO
            tok, smargin, mass = inverse_cdf(p_m, float(u_sample))
            mass = 0.0
    else:
        p_bonus = dist(target[gamma])
        tok, smargin, mass = inverse_cdf(p_bonus, float(u_sample))
    toks = [int(x) for x in drafts[:m]] + [tok]
    return SequenceResult(toks, m, status, gamma, False, p_d, q_d, mass, margins, smargin)


def verify_batch(target: np.ndarray, draft: Optional[np.ndarray], dtype: str,
                 draft_tokens: np.ndarray, num_draft: np.ndarray, temperature: Optional[np.ndarray],
                 u_accept: Optional[np.ndarray], u_sample: Optional[np.ndarray],
                 seqs=None, top_k: Optional[np.ndarray] = None,
                 top_p: Optional[np.ndarray] = None, nan_masked: bool = False) -> List[SequenceResult]:
    """Verify every sequence (or the listed ones) of a batch.

    target [B, gmax+1, V], draft [B, gmax, V] (bf16 bits or float32); a sequence whose
    temperature is not > 0, or every sequence when temperature is None, is greedy.
    """
    B, gp1, V = target.shape
    gmax = gp1 - 1
    out = []
    for b in (range(B) if seqs is None else seqs):
        g = int(num_draft[b])
        clamped = 0
        if g < 0 or g > gmax:
            g = min(max(g, 0), gmax)
            clamped = ST_CLAMPED_GAMMA
        P = widen(target[b, : g + 1], dtype)
        T = None if temperature is None else float(temperature[b])
        if T is None or not (T > 0.0):
            r = verify_greedy_sequence(P, draft_tokens[b], g)
        else:
            Q = widen(draft[b, :g], dtype) if g > 0 else np.zeros((0, V))
            r = verify_sample_sequence(P, Q, draft_tokens[b], g, T, u_accept[b], float(u_sample[b]),
                                       0 if top_k is None else int(top_k[b]),
                                       1.0 if top_p is None else float(top_p[b]), nan_masked)
        r.status |= clamped
        out.append(r)
    return out


def emitted_rows(results: List[SequenceResult], gmax: int) -> np.ndarray:
    """out_tokens layout [B, gmax+1]: the m+1 emitted tokens, then -1."""
    out = np.full((len(results), gmax + 1), -1, dtype=np.int64)
    for b, r in enumerate(results):
        out[b, : len(r.tokens)] = r.tokens
    return out


def commit_kv_lengths(kv_len: np.ndarray, m: np.ndarray, correction_processed: bool,
                      draft_kv_len: Optional[np.ndarray] = None, out_tokens: Optional[np.ndarray] = None,
                      history: Optional[np.ndarray] = None, committed_len: Optional[np.ndarray] = None):
    """Commit one round ([TUT] §5.1-§5.2; [KB] §06).

    Both caches are trimmed to t + m (the accepted prefix); once the correction or bonus
    token has been fed through both models they hold t + m + 1.  When a token history is
    given, the emitted tokens (out_tokens[b, :m+1] up to its first -1, which only a stop
    leaves there) are appended at committed_len; a sequence whose append position is not
    legal (committed_len < 0, or the history would overflow) is left untouched and flagged
    (bit 8).
    Returns (kv_len, draft_kv_len, history, committed_len, status) as new arrays.
    """
    kv = np.array(kv_len, dtype=np.int64)
    dkv = None if draft_kv_len is None else np.array(draft_kv_len, dtype=np.int64)
    hist = None if history is None else np.array(history)
    clen = None if committed_len is None else np.array(committed_len, dtype=np.int64)
    status = np.zeros(len(kv), dtype=np.int64)
    add = 1 if correction_processed else 0
    for b in range(len(kv)):
        n = int(m[b]) + 1
        if out_tokens is not None:
            # only the emitted tokens: a round cut by a stop leaves -1 after them
            lead = np.flatnonzero(np.asarray(out_tokens[b, :n]) < 0)
            if lead.size:
                n = int(lead[0])
        if hist is not None:
            cap = hist.shape[1]
            if clen[b] < 0 or clen[b] + n > cap:
                status[b] |= ST_HISTORY_FULL
                continue
            hist[b, clen[b]: clen[b] + n] = out_tokens[b, :n]
            clen[b] += n
        kv[b] += int(m[b]) + add
        if dkv is not None:
            dkv[b] += int(m[b]) + add
    return kv, dkv, hist, clen, status


def apply_stops(out_tokens: np.ndarray, m: np.ndarray, eos_id: int,
                max_new: Optional[np.ndarray] = None):
    """Cut each round's emit where step-by-step decoding would have stopped ([TUT] §5.2,
    §12.3; [KB] §03).

    The emit is out_tokens[b, :m+1] = d_0..d_{m-1}, tok.  It ends at its first token equal
    to eos_id (kept; eos_id < 0 means no end token) and holds at most max_new[b] tokens
    (the sequence's remaining budget; <= 0 emits nothing).  Emitted tokens stay, the rest
    become -1, and m becomes (tokens emitted) - 1, at least 0: every emitted token but the
    last has its cache entries kept, the last is fed next, as a correction token would be.
    Bit 32 marks a sequence that must not continue: its last emitted token is the end
    token, or its budget is used up.
    Returns (out_tokens, m, status) as new arrays.
    """
    out = np.array(out_tokens, dtype=np.int64)
    mm = np.array(m, dtype=np.int64)
    status = np.zeros(len(mm), dtype=np.int64)
    gmax = out.shape[1] - 1
    for b in range(len(mm)):
        n = min(max(int(mm[b]), 0), gmax) + 1
        if eos_id >= 0:
            hit = np.flatnonzero(out[b, :n] == eos_id)
            if hit.size:
                n = int(hit[0]) + 1
        stop_budget = False
        if max_new is not None:
            budget = int(max_new[b])
            n = min(n, max(budget, 0))
            stop_budget = n >= budget
        stop_eos = eos_id >= 0 and n >= 1 and out[b, n - 1] == eos_id
        out[b, n:] = -1
        mm[b] = max(n - 1, 0)
        if stop_eos or stop_budget:
            status[b] |= ST_STOPPED
    return out, mm, status


@dataclasses.dataclass
class TreeResult:
    tokens: List[int]   # the path's tokens, then the correction/bonus token
    path: List[int]     # accepted node indices along the path, root (0) excluded
    m: int              # path length = accepted drafts
    status: int
    n: int              # nodes after clamping


def verify_tree_greedy_sequence(target: np.ndarray, node_tokens: np.ndarray, node_parents: np.ndarray,
                                n: int) -> TreeResult:
    """Greedy verification of a draft tree ([TUT] §5.3).

    Nodes 1..n; node j carries token node_tokens[j-1] and has parent node_parents[j-1]
    (0 is the root, the position after the committed context).  target: float64
    [>= n+1, V]; row j is the target's prediction for the position after node j.  Node j
    is accepted iff its parent is accepted (the root always is) and its token equals the
    argmax of its parent's row.  The path ends at the deepest accepted node (lowest index
    among equal depths); the step emits the path's tokens and then the argmax of that
    node's row -- the target's replacement where the tree ran out of matching drafts, or
    its bonus token at a leaf.
    """
    V = target.shape[1]
    status = 0
    accepted = [True] + [False] * n
    depth = [0] * (n + 1)
    best = 0
    for j in range(1, n + 1):
        par = int(node_parents[j - 1])
        d = int(node_tokens[j - 1])
        if not (0 <= par < j):
            status |= ST_BAD_TREE
            continue
        depth[j] = depth[par] + 1
        if not accepted[par]:
            continue
        if not (0 <= d < V):
            status |= ST_BAD_DRAFT
            continue
        if d == greedy_argmax(target[par]):
            accepted[j] = True
            if depth[j] > depth[best]:
                best = j
    path = []
    j = best
    while j != 0:
        path.append(j)
        j = int(node_parents[j - 1])
    path.reverse()
    tokens = [int(node_tokens[c - 1]) for c in path] + [greedy_argmax(target[best])]
    return TreeResult(tokens, path, len(path), status, n)


def verify_tree_batch(target: np.ndarray, dtype: str, node_tokens: np.ndarray, node_parents: np.ndarray,
                      num_nodes: Optional[np.ndarray], seqs=None) -> List[TreeResult]:
    """Greedy tree verification of every sequence (or the listed ones): target
    [B, nmax+1, V], node_tokens and node_parents [B, nmax]; num_nodes [B] (None: nmax),
    clamped to [0, nmax] with status bit 4."""
    B, np1, V = target.shape
    nmax = np1 - 1
    out = []
    for b in (range(B) if seqs is None else seqs):
        n = nmax if num_nodes is None else int(num_nodes[b])
        clamped = 0
        if n < 0 or n > nmax:
            n = min(max(n, 0), nmax)
            clamped = ST_CLAMPED_GAMMA
        r = verify_tree_greedy_sequence(widen(target[b, : n + 1], dtype), node_tokens[b], node_parents[b], n)
        r.status |= clamped
        out.append(r)
    return out
