"""Seeded synthetic inputs for the batched verify-and-commit step.

This module only draws random numbers: target and draft logits, the draft
tokens a proposer would have produced, the explicit uniforms the verifier
consumes, per-sequence draft lengths and pre-round KV lengths.  It holds none
of the verification arithmetic (no softmax, no acceptance test, no residual,
no inverse CDF), so both the CUDA path and the float64 oracle can be fed from
it without sharing any of the method.

Drafting itself lies outside the verify step (it is the proposer's job in the
"draft -> verify -> accept/reject -> commit" round of the tutorial
"投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡", §2-§3.1).  The
proposer here samples a draft token from softmax(Q/T) with the Gumbel-max
trick, argmax_v(Q_v/T + G_v) with G_v ~ Gumbel(0,1), or takes argmax_v Q_v when
it decodes greedily.  It never looks at the target logits P, except in the
greedy workload where the target argmax is *planted* (the generator chooses it
first and writes a strict maximum there) instead of being computed.

Layouts (row-major, contiguous):
  target  [B, gmax+1, V]   row i judges draft i; row 0 is the saved boundary
                           prediction; row num_draft[b] is the bonus row
  draft   [B, gmax, V]     draft logits, row i is the distribution draft i came from
  draft_tokens [B, gmax] int32, padding (i >= num_draft[b]) is -1
  logits past a sequence's last valid row are NaN, so a stray read shows.

bf16 tensors are carried as uint16 bit patterns (numpy has no bf16 type),
rounded from float32 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    r[np.isnan(x)] = BF16_NAN
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                      # "bf16" (uint16 bits) or "f32"
    B: int
    gmax: int
    V: int
    target: np.ndarray              # [B, gmax+1, V]
    draft: Optional[np.ndarray]     # [B, gmax, V] or None (greedy-only workload)
    draft_tokens: np.ndarray        # int32 [B, gmax]
    num_draft: np.ndarray           # int32 [B]
    temperature: np.ndarray         # float32 [B]; <= 0 means a greedy sequence
    u_accept: np.ndarray            # float32 [B, gmax] in [0, 1)
    u_sample: np.ndarray            # float32 [B] in [0, 1)
    kv_len: np.ndarray              # int32 [B], pre-round committed KV length t
    greedy_only: bool = False

    def verified_rows(self) -> int:
        """Draft rows judged per call: sum over sequences of num_draft."""
        return int(self.num_draft.sum())

    def algorithmic_bytes(self) -> int:
        """Bytes of logits the step must read once: every valid target row, plus
        the draft rows of sampling sequences."""
        es = 2 if self.dtype == "bf16" else 4
        g = self.num_draft.astype(np.int64)
        sampling = (self.temperature > 0) & (not self.greedy_only)
        rows = int((g + 1).sum() + g[sampling].sum())
        return rows * self.V * es


def _streams(cfg: int, seed: int, n: int):
    ss = np.random.SeedSequence([2026, cfg, seed])
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def _gumbel_draft(rng: np.random.Generator, q_logits: np.ndarray, T: float) -> int:
    """Proposer: sample one token from softmax(q_logits / T) by Gumbel-max."""
    g = rng.gumbel(size=q_logits.shape[0])
    return int(np.argmax(q_logits.astype(np.float64) / T + g))


def _pack(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == "bf16" else x32.astype(np.float32)


def _unpack(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x) if dtype == "bf16" else x


def _alloc(shape, dtype):
    if dtype == "bf16":
        return np.full(shape, BF16_NAN, dtype=np.uint16)
    return np.full(shape, np.nan, dtype=np.float32)


def sampling_workload(name: str, *, cfg: int, seed: int, B: int, gmax: int, V: int,
                      dtype: str, target_sigma: float, draft_scale: float,
                      draft_sigma, temperature, boost_frac: float = 0.0,
                      boost: float = 0.0, num_draft=None, greedy_mask=None,
                      equal_mask=None, kv_range=(512, 8192)) -> Workload:
    """Generic sampling (or mixed) workload.

    target row  ~ N(0, target_sigma^2), plus `boost` on round(boost_frac*V) distinct ids
    draft row   = draft_scale * target + N(0, sigma_b^2), sigma_b = draft_sigma[b]
    equal_mask[b] -> draft rows are bit-identical to the target rows (q == p)
    greedy_mask[b] -> temperature 0 and greedy drafts argmax(draft row)
    """
    (r_t, r_n, r_d, r_ua, r_us, r_g, r_b, r_kv) = _streams(cfg, seed, 8)
    if num_draft is None:
        num_draft = np.full(B, gmax, dtype=np.int32)
    num_draft = np.asarray(num_draft, dtype=np.int32)
    sig = np.broadcast_to(np.asarray(draft_sigma, dtype=np.float64), (B,))
    temp = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)).copy()
    greedy_mask = np.zeros(B, bool) if greedy_mask is None else np.asarray(greedy_mask, bool)
    equal_mask = np.zeros(B, bool) if equal_mask is None else np.asarray(equal_mask, bool)
    temp[greedy_mask] = 0.0

    tgt = _alloc((B, gmax + 1, V), dtype)
    drf = _alloc((B, gmax, V), dtype)
    toks = np.full((B, gmax), -1, dtype=np.int32)
    n_boost = int(round(boost_frac * V))
    for b in range(B):
        g = int(num_draft[b])
        t32 = (r_t.standard_normal((g + 1, V), dtype=np.float32) * np.float32(target_sigma))
        if n_boost:
            for i in range(g + 1):
                ids = r_b.choice(V, size=n_boost, replace=False)
                t32[i, ids] += np.float32(boost)
        tgt[b, : g + 1] = _pack(t32, dtype)
        if g == 0:
            continue
        if equal_mask[b]:
            drf[b, :g] = tgt[b, :g]
        else:
            noise = r_n.standard_normal((g, V), dtype=np.float32) * np.float32(sig[b])
            drf[b, :g] = _pack(np.float32(draft_scale) * t32[:g] + noise, dtype)
        qv = _unpack(drf[b, :g], dtype)
        for i in range(g):
            if greedy_mask[b]:
                toks[b, i] = int(np.argmax(qv[i]))
            else:
                toks[b, i] = _gumbel_draft(r_d, qv[i], float(temp[b]))
    ua = r_ua.random((B, gmax), dtype=np.float32)
    us = r_us.random(B, dtype=np.float32)
    kv = r_kv.integers(kv_range[0], kv_range[1] + 1, size=B).astype(np.int32)
    return Workload(name, dtype, B, gmax, V, tgt, drf, toks, num_draft, temp, ua, us, kv)


def greedy_planted_workload(name: str, *, cfg: int, seed: int, B: int, gmax: int, V: int,
                            sigma: float = 3.0, alpha: float = 0.8) -> Workload:
    """Greedy workload with a planted target argmax.

    Each target row is N(0, sigma^2) clipped to +-6 sigma, and the generator
    writes 6 sigma + 1 at a uniformly chosen id g (so g is the unique argmax by
    construction).  Draft i equals g_i with probability alpha, else a uniform
    id other than g_i.  No draft logits are produced (greedy verification reads
    none).
    """
    (r_t, r_g, r_a, r_o, r_kv) = _streams(cfg, seed, 5)
    hi = np.float32(6.0 * sigma)
    tgt = np.empty((B, gmax + 1, V), dtype=np.uint16)
    planted = r_g.integers(0, V, size=(B, gmax + 1))
    for b in range(B):
        t32 = np.clip(r_t.standard_normal((gmax + 1, V), dtype=np.float32) * np.float32(sigma), -hi, hi)
        t32[np.arange(gmax + 1), planted[b]] = hi + np.float32(1.0)
        tgt[b] = f32_to_bf16_bits(t32)
    match = r_a.random((B, gmax)) < alpha
    other = r_o.integers(0, V - 1, size=(B, gmax))
    pl = planted[:, :gmax]
    other = other + (other >= pl)
    toks = np.where(match, pl, other).astype(np.int32)
    num_draft = np.full(B, gmax, dtype=np.int32)
    kv = r_kv.integers(512, 8193, size=B).astype(np.int32)
    return Workload(name, "bf16", B, gmax, V, tgt, None, toks, num_draft,
                    np.zeros(B, np.float32), np.zeros((B, gmax), np.float32),
                    np.zeros(B, np.float32), kv, greedy_only=True)


def three_token_workload(B: int, seed: int = 0) -> Workload:
    """The three-token worked example p=(0.5,0.3,0.2), q=(0.2,0.5,0.3), one draft
    per sequence, logits ln p / ln q in float32, bonus row ln p, T = 1, drafts
    drawn from q.  B independent trials in one batch."""
    (r_d, r_ua, r_us) = _streams(1003, seed, 3)
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.5, 0.3])
    lp = np.log(p).astype(np.float32)
    lq = np.log(q).astype(np.float32)
    tgt = np.broadcast_to(lp, (B, 2, 3)).copy()
    drf = np.broadcast_to(lq, (B, 1, 3)).copy()
    toks = r_d.choice(3, size=(B, 1), p=q).astype(np.int32)
    ua = r_ua.random((B, 1), dtype=np.float32)
    us = r_us.random(B, dtype=np.float32)
    return Workload("three-token", "f32", B, 1, 3, tgt, drf, toks, np.ones(B, np.int32),
                    np.ones(B, np.float32), ua, us, np.full(B, 100, np.int32))


# ----------------------------------------------------------------------------------------
# The five named workloads.  Sizes and distributions follow the workload table of the
# verify-and-commit study; where it leaves a detail open the reading is stated inline.
# ----------------------------------------------------------------------------------------

def small_fp32(seed: int = 0) -> Workload:
    """B=8, gamma=4, V=1024, fp32 target ~ N(0,2^2), draft = target + N(0,0.5^2), T=1."""
    return sampling_workload("small-fp32-B8-g4-V1024", cfg=1, seed=seed, B=8, gmax=4, V=1024,
                             dtype="f32", target_sigma=2.0, draft_scale=1.0, draft_sigma=0.5,
                             temperature=1.0)


def greedy_32k(seed: int = 0) -> Workload:
    """Greedy: B=64, gamma=5, V=32000, bf16 ~ N(0,3^2), drafts match the argmax w.p. 0.8."""
    return greedy_planted_workload("greedy-B64-g5-V32000", cfg=2, seed=seed, B=64, gmax=5, V=32000)


def sampling_128k(seed: int = 0) -> Workload:
    """Sampling: B=128, gamma=4, V=128256, bf16 target ~ N(0,3^2) with 1% of ids (1283,
    distinct per row) boosted by +8; draft = 0.7*target + N(0,1); T=0.8 both sides."""
    return sampling_workload("sampling-B128-g4-V128256-bf16", cfg=3, seed=seed, B=128, gmax=4,
                             V=128256, dtype="bf16", target_sigma=3.0, draft_scale=0.7,
                             draft_sigma=1.0, temperature=0.8, boost_frac=0.01, boost=8.0)


def mixed_152k(seed: int = 0) -> Workload:
    """Mixed: B=256, V=151936, bf16, gamma_b ~ U{1..8} padded to 8; even b greedy, odd b
    sampling at T=0.7; target ~ N(0,3^2) (the sigma the other workloads use); draft =
    target + N(0,1.5^2); t ~ U{512..8192}."""
    rng = _streams(4, seed, 9)[8]
    g = rng.integers(1, 9, size=256).astype(np.int32)
    greedy = (np.arange(256) % 2) == 0
    return sampling_workload("mixed-B256-g1..8-V151936-bf16", cfg=4, seed=seed, B=256, gmax=8,
                             V=151936, dtype="bf16", target_sigma=3.0, draft_scale=1.0,
                             draft_sigma=1.5, temperature=0.7, num_draft=g, greedy_mask=greedy)


def large_batch_128k(seed: int = 0, B: int = 1024) -> Workload:
    """Large batch: B=1024, gamma=4, V=128256, bf16 ~ N(0,3^2); draft = target +
    N(0,sigma_b^2), sigma_b ~ U[0.2,3]; every 16th sequence has q == p exactly; T=1."""
    rng = _streams(5, seed, 9)[8]
    sig = rng.uniform(0.2, 3.0, size=B)
    eq = (np.arange(B) % 16) == 0
    return sampling_workload(f"large-B{B}-g4-V128256-bf16", cfg=5, seed=seed, B=B, gmax=4,
                             V=128256, dtype="bf16", target_sigma=3.0, draft_scale=1.0,
                             draft_sigma=sig, temperature=1.0, equal_mask=eq)


@dataclasses.dataclass
class TreeWorkload:
    """Draft trees for greedy tree verification.  Node j (1..num_nodes[b]) carries
    node_tokens[b][j-1] and hangs below node_parents[b][j-1] < j (0 is the root)."""
    name: str
    dtype: str
    B: int
    nmax: int
    V: int
    target: np.ndarray              # [B, nmax+1, V]: row j follows node j
    node_tokens: np.ndarray         # int32 [B, nmax]
    node_parents: np.ndarray        # int32 [B, nmax]
    num_nodes: np.ndarray           # int32 [B]
    kv_len: np.ndarray              # int32 [B]

    def verified_rows(self) -> int:
        """Draft nodes judged per call."""
        return int(self.num_nodes.sum())

    def algorithmic_bytes(self) -> int:
        es = 2 if self.dtype == "bf16" else 4
        return int((self.num_nodes.astype(np.int64) + 1).sum()) * self.V * es


def tree_workload(name: str, *, cfg: int, seed: int, B: int, nmax: int, V: int, dtype: str = "bf16",
                  sigma: float = 3.0, alpha: float = 0.7, width: int = 4, num_nodes=None) -> TreeWorkload:
    """Draft trees with a planted target argmax.

    Node j's parent is uniform among nodes max(0, j-width)..j-1, so trees branch and deepen
    like the candidate trees of tree drafters.  Every target row is N(0, sigma^2) clipped to
    +-6 sigma, with 6 sigma + 1 written at a uniformly chosen id (its argmax by
    construction).  A node copies its parent row's planted id with probability alpha unless a
    sibling already holds it; otherwise it takes a uniform id that no sibling holds.  Rows past
    a sequence's node count are NaN.
    """
    (r_t, r_g, r_p, r_a, r_o, r_kv) = _streams(cfg, seed, 6)
    hi = np.float32(6.0 * sigma)
    n_arr = np.full(B, nmax, dtype=np.int32) if num_nodes is None else np.asarray(num_nodes, dtype=np.int32)
    tgt = _alloc((B, nmax + 1, V), dtype)
    toks = np.full((B, nmax), -1, dtype=np.int32)
    pars = np.full((B, nmax), -1, dtype=np.int32)
    for b in range(B):
        n = int(n_arr[b])
        t32 = np.clip(r_t.standard_normal((n + 1, V), dtype=np.float32) * np.float32(sigma), -hi, hi)
        planted = r_g.integers(0, V, size=n + 1)
        t32[np.arange(n + 1), planted] = hi + np.float32(1.0)
        tgt[b, : n + 1] = _pack(t32, dtype)
        taken = {}
        for j in range(1, n + 1):
            p = int(r_p.integers(max(0, j - width), j))
            sib = taken.setdefault(p, set())
            a = int(planted[p])
            if a not in sib and r_a.random() < alpha:
                t = a
            else:
                t = int(r_o.integers(0, V))
                while t == a or t in sib:
                    t = int(r_o.integers(0, V))
            sib.add(t)
            toks[b, j - 1] = t
            pars[b, j - 1] = p
    kv = r_kv.integers(512, 8193, size=B).astype(np.int32)
    return TreeWorkload(name, dtype, B, nmax, V, tgt, toks, pars, n_arr, kv)


def tree_63_128k(seed: int = 0) -> TreeWorkload:
    """Tree workload: B=32 sequences, 63-node draft trees, V=128256, bf16 ~ N(0,3^2) with a
    planted argmax per row; a node copies its parent's planted id with probability 0.7."""
    return tree_workload("tree-B32-n63-V128256-bf16", cfg=6, seed=seed, B=32, nmax=63, V=128256)


WORKLOADS = {1: small_fp32, 2: greedy_32k, 3: sampling_128k, 4: mixed_152k, 5: large_batch_128k, 6: tree_63_128k}
