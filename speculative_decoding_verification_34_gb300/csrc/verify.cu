// Fused greedy / sampling verification: one thread-block cluster per sequence.
//
// What is computed follows the tutorial "投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡"
// (§3-§4 greedy verification and logit alignment, §7.1-§7.3 acceptance min(1,p/q), residual
// max(p-q,0)/R and the bonus draw) and the "M013" knowledge-base card (§03-§05, including the
// R = 0 remark).  How it is computed is this library's own design for sm_103a:
//
//   * Cluster of C blocks per sequence b (C <= 16); block c owns the vocabulary chunk
//     [c*chunk, (c+1)*chunk) of every row of b.  Phase A streams the chunk of every row the
//     sequence needs once from HBM (128-bit loads, one exp2 per sampled element) and reduces
//     it to a (max, sum-of-exp) pair, or to an (argmax value, id) pair for greedy rows.
//   * Each block pushes its per-row partials into every block's shared memory (distributed
//     shared memory); after one cluster barrier every block holds all C partials and derives
//     the same row maxima/normalisers, the same acceptance flags and the same m.
//   * Phase B (sampling only): each block re-reads its chunk of the one row (pair) the final
//     draw needs -- row m of p and q after a rejection, the bonus row otherwise, normally
//     still in L2 -- and reduces the residual mass max(p-q,0) (and the p mass for the R = 0
//     fallback).  A second push + barrier gives every block all C chunk masses; the block
//     whose chunk holds u*R runs an in-chunk prefix scan to find the token and writes the
//     outputs.
//
// No global workspace, no atomics, no spin-waits: the only cross-block synchronisation is
// the hardware cluster barrier, reached by every block of a cluster the same number of times.

#include <cooperative_groups.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace specverify {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kQSlot = SPEC_MAX_GAMMA + 1;        // row slot of draft row i is kQSlot + i
constexpr int kSlots = kQSlot + SPEC_MAX_GAMMA;   // target rows 0..gmax, draft rows 0..gmax-1
constexpr int kVecPerPass = 4;                    // 16-byte vectors per thread per row per pass
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* num_draft;
  const float* temperature;
  const float* u_accept;
  const float* u_sample;
  int64_t V;
  int gmax;
  int chunk;
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* diag;
  int32_t* status;
};

// ------------------------------------------------------------------------------------------
// device helpers
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Streaming 128-bit read-only load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Tree sum into lane 0, then broadcast: every lane gets the same bits.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(kFull, v, o);
  return __shfl_sync(kFull, v, 0);
}

// (value, id) argmax with the lowest id winning ties.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(kFull, v, o);
    int i2 = __shfl_xor_sync(kFull, i, o);
    if (better(v2, i2, v, i)) { v = v2; i = i2; }
  }
}

// Merge two (max, sum of 2^((x-max)k)) partials; (-inf, 0) is the empty partial.  Products
// and sums are explicitly rounded (never contracted into FMAs) so that bit-identical target
// and draft rows always give bit-identical statistics.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float k) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  const float a = (m == -INFINITY) ? 0.f : __fmul_rn(s, ex2(__fmul_rn(m - M, k)));
  const float b = (m2 == -INFINITY) ? 0.f : __fmul_rn(s2, ex2(__fmul_rn(m2 - M, k)));
  m = M;
  s = __fadd_rn(a, b);
}

// p_v = 2^((x_v - M) k) / S, evaluated as ex2(x*k - M*k) * (1/S) with a rounded product.
__device__ __forceinline__ float prob(float x, float k, float mk, float inv_s) {
  return __fmul_rn(ex2(fmaf(x, k, -mk)), inv_s);
}

// max(p - q, 0) with a rounded difference: exactly 0 wherever p == q.
__device__ __forceinline__ float residual(float p, float q) { return fmaxf(__fsub_rn(p, q), 0.f); }

// Element formats.  A 16-byte vector holds kPerVec elements; -inf fills vectors past the end.
struct Bf16 {
  using raw = uint16_t;
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kNegInfPair = 0xff80ff80u;
  __device__ __forceinline__ static float at(const raw* row, int64_t i) {
    return __uint_as_float(uint32_t(__ldg(row + i)) << 16);
  }
  __device__ __forceinline__ static uint4 neg_inf() { return make_uint4(kNegInfPair, kNegInfPair, kNegInfPair, kNegInfPair); }
  __device__ __forceinline__ static float get(const uint4& v, int j) {
    const uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};

struct F32 {
  using raw = float;
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static float at(const raw* row, int64_t i) { return __ldg(row + i); }
  __device__ __forceinline__ static uint4 neg_inf() {
    const uint32_t n = 0xff800000u;
    return make_uint4(n, n, n, n);
  }
  __device__ __forceinline__ static float get(const uint4& v, int j) {
    return __uint_as_float(j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w);
  }
};

// One pass of one row: kVecPerPass vectors per thread, vector k of thread t at element
// e0 + (k*kThreads + t)*kPerVec (coalesced across the block for every k).
template <class E, bool kVec>
struct Tile {
  uint4 v[kVecPerPass];
  float s[kVec ? 1 : kVecPerPass * E::kPerVec];

  __device__ __forceinline__ void load(const typename E::raw* row, int64_t e0, int64_t hi, int tid) {
#pragma unroll
    for (int k = 0; k < kVecPerPass; ++k) {
      const int64_t e = e0 + int64_t(k * kThreads + tid) * E::kPerVec;
      if constexpr (kVec) {
        v[k] = e < hi ? ld_stream(row + e) : E::neg_inf();
      } else {
#pragma unroll
        for (int j = 0; j < E::kPerVec; ++j)
          s[k * E::kPerVec + j] = (e + j < hi) ? E::at(row, e + j) : -INFINITY;
      }
    }
  }
  __device__ __forceinline__ float x(int k, int j) const {
    if constexpr (kVec) return E::get(v[k], j);
    else return s[k * E::kPerVec + j];
  }
};

template <class E, bool kVec>
__device__ __forceinline__ void tile_stats(const Tile<E, kVec>& t, float k, float& run_m, float& run_s) {
  float m = -INFINITY;
#pragma unroll
  for (int a = 0; a < kVecPerPass; ++a)
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) m = fmaxf(m, t.x(a, j));
  m = warp_max(m);
  float s = 0.f;
  if (m != -INFINITY) {
    const float mk = __fmul_rn(m, k);
#pragma unroll
    for (int a = 0; a < kVecPerPass; ++a)
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j) s += ex2(fmaf(t.x(a, j), k, -mk));
  }
  s = warp_sum(s);
  merge_ms(run_m, run_s, m, s, k);
}

template <class E, bool kVec>
__device__ __forceinline__ void tile_argmax(const Tile<E, kVec>& t, int64_t e0, int tid, float& bv, int& bi) {
#pragma unroll
  for (int a = 0; a < kVecPerPass; ++a)
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) {
      const int idx = int(e0 + int64_t(a * kThreads + tid) * E::kPerVec + j);
      const float v = t.x(a, j);
      if (better(v, idx, bv, bi)) { bv = v; bi = idx; }
    }
}

struct Shared {
  float2 warp_part[kWarps][kSlots];   // per-warp partial of each row slot (this block)
  float2 local[kSlots];               // this block's chunk partial per row slot
  float2 all[kMaxCluster][kSlots];    // every block's chunk partials, pushed by their owners
  float2 mass_warp[kWarps];
  float2 all_mass[kMaxCluster];       // (weight mass, p mass) of every block's chunk
  float rowM[kSlots];                 // row max of the logits
  float rowInvS[kSlots];              // 1 / sum_v 2^((x_v - M) k)
  int rowArg[kSlots];                 // greedy argmax per target row
  float pd[SPEC_MAX_GAMMA], qd[SPEC_MAX_GAMMA];
  float scan_warp[kWarps];
  int m, g, flags, owner, cand, lastpos, token;
  float target_local, mass_out;
};

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------

template <class E, bool kVec, bool kMixed>
__global__ void __launch_bounds__(kThreads, 4) verify_kernel(const Args a) {
  using raw = typename E::raw;
  __shared__ Shared sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = int(cluster.num_blocks());
  const int rank = int(cluster.block_rank());
  const int b = int(blockIdx.x) / CL;
  const int tid = int(threadIdx.x);
  const int lane = tid & 31, warp = tid >> 5;

  // Split arrive: every block must be running before anyone writes into its shared memory.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  const int64_t V = a.V;
  const int gmax = a.gmax;
  int g = a.num_draft ? a.num_draft[b] : gmax;
  int flags = 0;
  if (g < 0 || g > gmax) {
    g = g < 0 ? 0 : gmax;
    flags |= SPEC_ST_CLAMPED_GAMMA;
  }
  float T = 0.f;
  if constexpr (kMixed) T = a.temperature[b];
  const bool sampling = kMixed && (T > 0.f);
  const float k = sampling ? kLog2e / T : 0.f;

  const raw* P = static_cast<const raw*>(a.target) + int64_t(b) * (gmax + 1) * V;
  const raw* Q = sampling ? static_cast<const raw*>(a.draft) + int64_t(b) * gmax * V : nullptr;
  const int64_t lo = int64_t(rank) * a.chunk;
  const int64_t hi = lo + a.chunk < V ? lo + a.chunk : V;
  constexpr int kPass = kThreads * kVecPerPass * E::kPerVec;

  // ---------------- phase A: one streaming pass over this block's chunk of every row -----
  if (sampling) {
    // bonus row alone, then (target_i, draft_i) pairs from i = g-1 down to 0 so that the
    // rows a rejection most often needs (small m) are the most recently read.
    for (int i = g; i >= 0; --i) {
      const raw* rp = P + int64_t(i) * V;
      const raw* rq = (i < g) ? Q + int64_t(i) * V : nullptr;
      float pm = -INFINITY, ps = 0.f, qm = -INFINITY, qs = 0.f;
      for (int64_t e0 = lo; e0 < hi; e0 += kPass) {
        Tile<E, kVec> tp, tq;
        tp.load(rp, e0, hi, tid);
        if (rq) tq.load(rq, e0, hi, tid);
        tile_stats(tp, k, pm, ps);
        if (rq) tile_stats(tq, k, qm, qs);
      }
      if (lane == 0) {
        sm.warp_part[warp][i] = make_float2(pm, ps);
        if (rq) sm.warp_part[warp][kQSlot + i] = make_float2(qm, qs);
      }
    }
  } else {
    for (int i = g; i >= 0; i -= 2) {
      const raw* r0 = P + int64_t(i) * V;
      const raw* r1 = (i >= 1) ? P + int64_t(i - 1) * V : nullptr;
      float v0 = -INFINITY, v1 = -INFINITY;
      int i0 = INT_MAX, i1 = INT_MAX;
      for (int64_t e0 = lo; e0 < hi; e0 += kPass) {
        Tile<E, kVec> t0, t1;
        t0.load(r0, e0, hi, tid);
        if (r1) t1.load(r1, e0, hi, tid);
        tile_argmax(t0, e0, tid, v0, i0);
        if (r1) tile_argmax(t1, e0, tid, v1, i1);
      }
      warp_argmax(v0, i0);
      if (r1) warp_argmax(v1, i1);
      if (lane == 0) {
        sm.warp_part[warp][i] = make_float2(v0, __int_as_float(i0));
        if (r1) sm.warp_part[warp][i - 1] = make_float2(v1, __int_as_float(i1));
      }
    }
  }
  __syncthreads();

  // block partial per row slot, warps merged in a fixed order
  const int nP = g + 1, nQ = sampling ? g : 0, nSlots = nP + nQ;
  for (int r = tid; r < nSlots; r += kThreads) {
    const int slot = r < nP ? r : kQSlot + (r - nP);
    float2 acc = sm.warp_part[0][slot];
    for (int w = 1; w < kWarps; ++w) {
      const float2 p = sm.warp_part[w][slot];
      if (sampling) {
        merge_ms(acc.x, acc.y, p.x, p.y, k);
      } else if (better(p.x, __float_as_int(p.y), acc.x, __float_as_int(acc.y))) {
        acc = p;
      }
    }
    sm.local[slot] = acc;
  }
  __syncthreads();

  // ---------------- exchange 1: push the partials into every block of the cluster --------
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (int idx = tid; idx < CL * nSlots; idx += kThreads) {
    const int c = idx / nSlots, r = idx - c * nSlots;
    const int slot = r < nP ? r : kQSlot + (r - nP);
    float2* dst = cluster.map_shared_rank(&sm.all[rank][slot], c);
    *dst = sm.local[slot];
  }
  cluster.sync();

  // every block combines the C partials of each row in the same order -> identical results
  for (int r = tid; r < nSlots; r += kThreads) {
    const int slot = r < nP ? r : kQSlot + (r - nP);
    if (sampling) {
      float M = -INFINITY;
      for (int c = 0; c < CL; ++c) M = fmaxf(M, sm.all[c][slot].x);
      float S = 0.f;
      if (M != -INFINITY)
        for (int c = 0; c < CL; ++c) {
          const float2 p = sm.all[c][slot];
          if (p.x != -INFINITY) S = __fadd_rn(S, __fmul_rn(p.y, ex2(__fmul_rn(p.x - M, k))));
        }
      sm.rowM[slot] = M;
      sm.rowInvS[slot] = __frcp_rn(S);
    } else {
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int c = 0; c < CL; ++c) {
        const float2 p = sm.all[c][slot];
        if (better(p.x, __float_as_int(p.y), bv, bi)) { bv = p.x; bi = __float_as_int(p.y); }
      }
      sm.rowArg[slot] = bi;
    }
  }
  __syncthreads();

  // ---------------- acceptance flags and the first rejection (warp 0) -----------------------
  if (warp == 0) {
    bool acc = false, valid = false;
    int d = -1;
    if (lane < g) {
      d = a.draft_tokens[int64_t(b) * gmax + lane];
      valid = d >= 0 && int64_t(d) < V;
      if (sampling) {
        float p = NAN, q = NAN;
        if (valid) {
          const float xp = E::at(P + int64_t(lane) * V, d);
          const float xq = E::at(Q + int64_t(lane) * V, d);
          p = prob(xp, k, __fmul_rn(sm.rowM[lane], k), sm.rowInvS[lane]);
          q = prob(xq, k, __fmul_rn(sm.rowM[kQSlot + lane], k), sm.rowInvS[kQSlot + lane]);
          const float u = a.u_accept[int64_t(b) * gmax + lane];
          // u < min(1, p/q): r = 0 when p = 0, r = +inf when q = 0 < p
          acc = (p == 0.f) ? (u < 0.f) : (p >= q ? (u < 1.f) : (__fmul_rn(u, q) < p));
        }
        sm.pd[lane] = p;
        sm.qd[lane] = q;
      } else {
        acc = valid && d == sm.rowArg[lane];
      }
    }
    const unsigned keep = __ballot_sync(kFull, acc);
    const unsigned rej = ~keep & (g >= 32 ? kFull : ((1u << g) - 1u));
    const int m = rej ? __ffs(rej) - 1 : g;
    const unsigned badmask = __ballot_sync(kFull, lane < g && !valid);
    if (lane == 0) {
      int f = flags;
      if (m < g && ((badmask >> m) & 1u)) f |= SPEC_ST_BAD_DRAFT;
      sm.m = m;
      sm.g = g;
      sm.flags = f;
    }
  }
  __syncthreads();
  const int m = sm.m;

  if (!sampling) {
    if (rank == 0) {
      for (int i = tid; i <= gmax; i += kThreads) {
        int v = -1;
        if (i < m) v = a.draft_tokens[int64_t(b) * gmax + i];
        else if (i == m) v = sm.rowArg[m];
        a.out_tokens[int64_t(b) * (gmax + 1) + i] = v;
      }
      if (a.diag)
        for (int i = tid; i < 2 * gmax + 1; i += kThreads) a.diag[int64_t(b) * (2 * gmax + 1) + i] = NAN;
      if (tid == 0) {
        a.num_accepted[b] = m;
        if (a.status) a.status[b] = sm.flags;
      }
    }
    return;
  }

  // ---------------- phase B: chunk mass of the distribution the last token is drawn from ---
  const bool pair = m < g;                 // rejection: residual of (p_m, q_m); else bonus p_g
  const raw* rp = P + int64_t(m) * V;
  const raw* rq = pair ? Q + int64_t(m) * V : nullptr;
  const float mkp = __fmul_rn(sm.rowM[m], k), invp = sm.rowInvS[m];
  const float mkq = pair ? __fmul_rn(sm.rowM[kQSlot + m], k) : 0.f;
  const float invq = pair ? sm.rowInvS[kQSlot + m] : 0.f;
  float wsum = 0.f, psum = 0.f;
  for (int64_t e0 = lo; e0 < hi; e0 += kPass) {
    Tile<E, kVec> tp, tq;
    tp.load(rp, e0, hi, tid);
    if (pair) tq.load(rq, e0, hi, tid);
#pragma unroll
    for (int x = 0; x < kVecPerPass; ++x)
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j) {
        const float p = prob(tp.x(x, j), k, mkp, invp);
        psum += p;
        if (pair) wsum += residual(p, prob(tq.x(x, j), k, mkq, invq));
      }
  }
  if (!pair) wsum = psum;
  wsum = warp_sum(wsum);
  psum = warp_sum(psum);
  if (lane == 0) sm.mass_warp[warp] = make_float2(wsum, psum);
  __syncthreads();
  if (tid < CL) {
    float2 acc = sm.mass_warp[0];
    for (int w = 1; w < kWarps; ++w) { acc.x += sm.mass_warp[w].x; acc.y += sm.mass_warp[w].y; }
    float2* dst = cluster.map_shared_rank(&sm.all_mass[rank], tid);
    *dst = acc;
  }
  cluster.sync();

  // ---------------- which chunk holds u * total (every block, same order) ------------------
  if (tid == 0) {
    float R = 0.f, Pm = 0.f;
    for (int c = 0; c < CL; ++c) { R += sm.all_mass[c].x; Pm += sm.all_mass[c].y; }
    const bool use_w = !pair || R > 0.f;   // bonus: w is p itself
    int f = sm.flags;
    if (!use_w) f |= SPEC_ST_R_ZERO;
    const float total = use_w ? R : Pm;
    const float target = a.u_sample[b] * total;
    int owner = -1, last = 0;
    float excl = 0.f, run = 0.f;
    for (int c = 0; c < CL; ++c) {
      const float w = use_w ? sm.all_mass[c].x : sm.all_mass[c].y;
      if (w > 0.f) last = c;
      if (owner < 0) {
        excl = run;
        run += w;
        if (run > target && w > 0.f) owner = c;
      }
    }
    if (owner < 0) { owner = last; excl = 0.f; for (int c = 0; c < last; ++c) excl += use_w ? sm.all_mass[c].x : sm.all_mass[c].y; }
    sm.owner = owner;
    sm.flags = f | (use_w ? 0 : 0x100);   // 0x100: draw from p (internal)
    sm.target_local = target - excl;
    sm.mass_out = pair ? (use_w ? R : 0.f) : R;
    sm.cand = INT_MAX;
    sm.lastpos = -1;
  }
  __syncthreads();
  if (rank != sm.owner) return;

  // ---------------- owner block: prefix scan inside the chunk ------------------------------
  const bool draw_p = !pair || (sm.flags & 0x100);
  const float tl = sm.target_local;
  int64_t seg = (hi - lo + kThreads - 1) / kThreads;
  seg = (seg + E::kPerVec - 1) / E::kPerVec * E::kPerVec;
  const int64_t s0 = lo + int64_t(tid) * seg;
  const int64_t s1 = (s0 + seg < hi) ? s0 + seg : hi;
  auto weight = [&](int64_t v) -> float {
    const float p = prob(E::at(rp, v), k, mkp, invp);
    if (draw_p) return p;
    return residual(p, prob(E::at(rq, v), k, mkq, invq));
  };
  float mysum = 0.f;
  int mylast = -1;
  for (int64_t v = s0; v < s1; ++v) {
    const float w = weight(v);
    mysum += w;
    if (w > 0.f) mylast = int(v);
  }
  // block exclusive scan of the per-thread sums (warp scan, then warp totals in order)
  float incl = mysum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.scan_warp[warp] = incl;
  __syncthreads();
  float woff = 0.f;
  for (int w = 0; w < warp; ++w) woff += sm.scan_warp[w];
  const float excl = woff + incl - mysum;
  if (mysum > 0.f && excl + mysum > tl) atomicMin(&sm.cand, tid);
  if (mylast >= 0) atomicMax(&sm.lastpos, mylast);
  __syncthreads();
  if (tid == sm.cand) {
    int tok = mylast;
    float r = excl;
    for (int64_t v = s0; v < s1; ++v) {
      const float w = weight(v);
      r += w;
      if (w > 0.f && r > tl) { tok = int(v); break; }
    }
    sm.token = tok;
  }
  if (tid == 0 && sm.cand == INT_MAX) sm.token = sm.lastpos >= 0 ? sm.lastpos : int(lo);
  __syncthreads();

  const int tok = sm.token;
  for (int i = tid; i <= gmax; i += kThreads) {
    int v = -1;
    if (i < m) v = a.draft_tokens[int64_t(b) * gmax + i];
    else if (i == m) v = tok;
    a.out_tokens[int64_t(b) * (gmax + 1) + i] = v;
  }
  if (a.diag) {
    float* dg = a.diag + int64_t(b) * (2 * gmax + 1);
    for (int i = tid; i < gmax; i += kThreads) {
      dg[2 * i] = i < g ? sm.pd[i] : NAN;
      dg[2 * i + 1] = i < g ? sm.qd[i] : NAN;
    }
    if (tid == 0) dg[2 * gmax] = sm.mass_out;
  }
  if (tid == 0) {
    a.num_accepted[b] = m;
    if (a.status) a.status[b] = sm.flags & 0xff;
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

struct Plan {
  int cl;
  int chunk;
};

Plan make_plan(int64_t V) {
  int cl = int((V + 4095) / 4096);
  if (cl < 1) cl = 1;
  if (cl > kMaxCluster) cl = kMaxCluster;
  int64_t c = (V + cl - 1) / cl;
  c = (c + 7) / 8 * 8;
  return Plan{cl, int(c)};
}

std::mutex g_attr_mu;

template <class E, bool kVec, bool kMixed>
int launch(const Args& args, int B, void* stream) {
  auto fn = verify_kernel<E, kVec, kMixed>;
  const Plan plan = make_plan(args.V);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  {
    // cluster sizes above 8 need an opt-in; done once per device and kernel
    static bool done[64] = {};
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 64 && !done[dev]) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(NonPortableClusterSizeAllowed)");
      done[dev] = true;
    }
  }
  if (int64_t(B) * plan.cl > INT_MAX) {
    set_error("B=%d too large for %d blocks per sequence", B, plan.cl);
    return SPEC_ENOSPACE;
  }
  Args a = args;
  a.chunk = plan.chunk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B * plan.cl), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(plan.cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fn, a);
  if (e != cudaSuccess) return cuda_fail(e, "verify kernel launch");
  count_launch();
  return SPEC_OK;
}

int check_common(const void* target, int dtype, const int32_t* draft_tokens, int B, int gmax, int V,
                 int32_t* out_tokens, int32_t* num_accepted) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) {
    set_error("unknown dtype code %d", dtype);
    return SPEC_EDTYPE;
  }
  if (B < 0 || V < 1 || V > (1 << 30) || gmax < 0) {
    set_error("bad sizes B=%d gmax=%d V=%d", B, gmax, V);
    return SPEC_EINVAL;
  }
  if (gmax > SPEC_MAX_GAMMA) {
    set_error("gmax=%d exceeds SPEC_MAX_GAMMA=%d", gmax, SPEC_MAX_GAMMA);
    return SPEC_ENOSPACE;
  }
  if (B == 0) return SPEC_OK;   // empty batch: nothing is read or written, pointers may be null
  if (!target || !out_tokens || !num_accepted || (gmax > 0 && !draft_tokens)) {
    set_error("null required pointer");
    return SPEC_EINVAL;
  }
  return SPEC_OK;
}

bool vec_ok(const void* p, int dtype, int64_t V) {
  const int64_t es = dtype == SPEC_BF16 ? 2 : 4;
  return p == nullptr || ((reinterpret_cast<uintptr_t>(p) % 16 == 0) && (V * es) % 16 == 0);
}

}  // namespace
}  // namespace specverify

using namespace specverify;

namespace {
template <bool kMixed>
int dispatch_on(const Args& a, int dtype, int B, void* stream) {
  const bool vec = vec_ok(a.target, dtype, a.V) && vec_ok(a.draft, dtype, a.V);
  if (dtype == SPEC_BF16)
    return vec ? launch<Bf16, true, kMixed>(a, B, stream) : launch<Bf16, false, kMixed>(a, B, stream);
  return vec ? launch<F32, true, kMixed>(a, B, stream) : launch<F32, false, kMixed>(a, B, stream);
}
}  // namespace

extern "C" int spec_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens,
                                  const int32_t* num_draft, int B, int gmax, int V,
                                  int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                                  void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK) return rc;
  if (B == 0) return SPEC_OK;
  Args a = {};
  a.target = target_logits;
  a.draft_tokens = draft_tokens;
  a.num_draft = num_draft;
  a.V = V;
  a.gmax = gmax;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.status = status;
  return dispatch_on<false>(a, dtype, B, stream);
}

extern "C" int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                                  const int32_t* draft_tokens, const int32_t* num_draft,
                                  const float* temperature, const float* u_accept,
                                  const float* u_sample, int B, int gmax, int V,
                                  int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                  int32_t* status, void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK) return rc;
  if (B > 0 && (!temperature || !u_sample || (gmax > 0 && (!draft_logits || !u_accept)))) {
    set_error("null required pointer (draft_logits, temperature, u_accept or u_sample)");
    return SPEC_EINVAL;
  }
  if (B == 0) return SPEC_OK;
  Args a = {};
  a.target = target_logits;
  a.draft = draft_logits;
  a.draft_tokens = draft_tokens;
  a.num_draft = num_draft;
  a.temperature = temperature;
  a.u_accept = u_accept;
  a.u_sample = u_sample;
  a.V = V;
  a.gmax = gmax;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.diag = diag;
  a.status = status;
  return dispatch_on<true>(a, dtype, B, stream);
}

extern "C" int spec_verify_plan(int V, int dtype, int* ctas_per_seq, int* chunk) {
  clear_error();
  if (V < 1 || (dtype != SPEC_BF16 && dtype != SPEC_F32) || !ctas_per_seq || !chunk) {
    set_error("bad arguments to spec_verify_plan");
    return SPEC_EINVAL;
  }
  const Plan p = make_plan(V);
  *ctas_per_seq = p.cl;
  *chunk = p.chunk;
  return SPEC_OK;
}
