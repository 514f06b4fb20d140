// Fused greedy / sampling verification: one thread-block cluster per sequence.
//
// What is computed follows the tutorial "投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡"
// (§3-§4 greedy verification and logit alignment, §7.1-§7.3 acceptance min(1,p/q), residual
// max(p-q,0)/R and the bonus draw) and the "M013" knowledge-base card (§03-§05, including the
// R = 0 remark).  How it is computed is this library's own design for sm_103a:
//
//   * Cluster of C blocks per sequence b (C <= 16); block c owns the vocabulary chunk
//     [c*chunk, (c+1)*chunk) of every row of b.
//   * Phase A streams the chunk of every row the sequence needs exactly once from HBM.  Each
//     thread keeps its own 16-byte vectors in flight through a kStages-deep ring in shared
//     memory (cp.async, one commit group per tile), so loads of the next tiles overlap the
//     arithmetic on the current one.  A tile reduces to a (max, sum 2^((x-max)k)) pair with one
//     ex2 per element (bf16x2 max, f32x2 FMA/ADD), or to (max, lowest id) for greedy rows.
//   * Exchange 1: every block pushes its per-row partials into every block's shared memory
//     (distributed shared memory); after one cluster barrier all blocks derive, in the same
//     order, the same row maxima/normalisers, acceptance flags and m.
//   * Phase B (sampling only): every block re-reads its chunk of the row (pair) the last token
//     is drawn from -- row m of p and q after a rejection, the bonus row otherwise; normally an
//     L2 hit -- keeping one partial sum per (pass, vector slot, thread) in shared memory, and
//     pushes its chunk mass (exchange 2, second cluster barrier).
//   * The block whose chunk holds u*R finds the token from its per-vector sums (warp scans,
//     one vector reloaded) and writes the outputs.
//
// No global workspace, no atomics on global memory, no spin-waits: the only cross-block
// synchronisation is the hardware cluster barrier, which every block of a cluster reaches the
// same number of times.  cp.async groups are waited per thread (the thread's own copies).

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace specverify {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kVecPerPass = 8;                         // 16-byte vectors per thread per tile
constexpr int kStages = 3;                             // cp.async ring depth (tiles)
constexpr int kTileBytes = kThreads * kVecPerPass * 16;
constexpr int kMaxSlices = 128;                        // (pass, vector slot) pairs per chunk
constexpr int kMaxDynSmem = 160 * 1024;
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

// Packed pairs of f32 (sm_100+ f32x2 arithmetic), all round-to-nearest, never contracted.
using f2 = unsigned long long;
__device__ __forceinline__ f2 pk(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 upk(f2 r) {
  float2 v;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 ex2x2(f2 a) {
  const float2 v = upk(a);
  return pk(ex2(v.x), ex2(v.y));
}

// 16-byte global -> shared copy that bypasses L1; src_bytes = 0 zero-fills without reading.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 ld_l2(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Warp-wide max in one instruction (sm_100+ f32 redux); -inf is the identity.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Tree sum into lane 0, then broadcast: every lane gets the same bits.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_down_sync(kFull, v, o));
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
// and sums are explicitly rounded so bit-identical rows always give bit-identical statistics.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float k) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  const float a = (m == -INFINITY) ? 0.f : __fmul_rn(s, ex2(__fmul_rn(m - M, k)));
  const float b = (m2 == -INFINITY) ? 0.f : __fmul_rn(s2, ex2(__fmul_rn(m2 - M, k)));
  m = M;
  s = __fadd_rn(a, b);
}

// p_v = 2^((x_v - M) k) / S, evaluated as ex2(x*k - M*k) * (1/S) with a rounded product.
// prob() and prob2() give identical bits for the same element.
__device__ __forceinline__ float prob(float x, float k, float mk, float inv_s) {
  return __fmul_rn(ex2(fmaf(x, k, -mk)), inv_s);
}
__device__ __forceinline__ f2 prob2(f2 x, f2 k2, f2 nmk2, f2 inv2) { return mul2(ex2x2(fma2(x, k2, nmk2)), inv2); }

// max(p - q, 0) with a rounded difference: exactly 0 wherever p == q.
__device__ __forceinline__ float residual(float p, float q) { return fmaxf(__fsub_rn(p, q), 0.f); }

// Element formats.  A 16-byte vector holds kPerVec elements.
struct Bf16 {
  using raw = uint16_t;
  static constexpr int kPerVec = 8;
  __device__ __forceinline__ static float at(const raw* row, int64_t i) {
    return __uint_as_float(uint32_t(__ldg(row + i)) << 16);
  }
  // element pair j (0..3) of a vector, widened to f32x2 (lower id first)
  __device__ __forceinline__ static f2 pair(const uint4& v, int j) {
    const uint32_t w = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
    return pk(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ __forceinline__ static float get(const uint4& v, int j) {
    const uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  static constexpr uint32_t kNegInf = 0xff80ff80u;   // two bf16 -inf
  // max over kVecPerPass vectors: bf16x2 max tree, one widening at the end
  __device__ __forceinline__ static float tmax(const uint4 (&v)[kVecPerPass]) {
    __nv_bfloat162 a[kVecPerPass];
#pragma unroll
    for (int q = 0; q < kVecPerPass; ++q) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
      a[q] = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    }
#pragma unroll
    for (int w = kVecPerPass / 2; w > 0; w >>= 1)
#pragma unroll
      for (int q = 0; q < w; ++q) a[q] = __hmax2(a[q], a[q + w]);
    return fmaxf(__low2float(a[0]), __high2float(a[0]));
  }
};

struct F32 {
  using raw = float;
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static float at(const raw* row, int64_t i) { return __ldg(row + i); }
  __device__ __forceinline__ static f2 pair(const uint4& v, int j) {
    return j == 0 ? pk(__uint_as_float(v.x), __uint_as_float(v.y)) : pk(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ __forceinline__ static float get(const uint4& v, int j) {
    return __uint_as_float(j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w);
  }
  static constexpr uint32_t kNegInf = 0xff800000u;
  __device__ __forceinline__ static float tmax(const uint4 (&v)[kVecPerPass]) {
    float a[kVecPerPass];
#pragma unroll
    for (int q = 0; q < kVecPerPass; ++q)
      a[q] = fmaxf(fmaxf(__uint_as_float(v[q].x), __uint_as_float(v[q].y)),
                   fmaxf(__uint_as_float(v[q].z), __uint_as_float(v[q].w)));
#pragma unroll
    for (int w = kVecPerPass / 2; w > 0; w >>= 1)
#pragma unroll
      for (int q = 0; q < w; ++q) a[q] = fmaxf(a[q], a[q + w]);
    return a[0];
  }
};

// A tile is one pass of one row: vector k of thread t covers elements
// e0 + (k*kThreads + t)*kPerVec .. +kPerVec-1 (coalesced across the block for every k).
// Vector path: the vectors come from the shared-memory ring.  Scalar path (unaligned rows):
// elements are loaded one by one.  Out-of-range elements read as -inf.
template <class E, bool kVec>
struct Tile {
  static constexpr int N = E::kPerVec;
  uint4 v[kVecPerPass];
  float s[kVec ? 1 : kVecPerPass * N];

  // vector path: vectors q >= nq of this thread lie past the chunk end -> -inf
  __device__ __forceinline__ void mask_tail(int nq) {
    if constexpr (kVec) {
#pragma unroll
      for (int q = 0; q < kVecPerPass; ++q)
        if (q >= nq) v[q] = make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
    }
  }
  __device__ __forceinline__ float x(int k, int j) const {
    if constexpr (kVec) return E::get(v[k], j);
    else return s[k * N + j];
  }
};

template <class E, bool kVec>
__device__ __forceinline__ void tile_stats(const Tile<E, kVec>& t, float k, float& run_m, float& run_s) {
  constexpr int N = E::kPerVec;
  float m;
  if constexpr (kVec) {
    m = E::tmax(t.v);
  } else {
    m = -INFINITY;
#pragma unroll
    for (int a = 0; a < kVecPerPass * N; ++a) m = fmaxf(m, t.s[a]);
  }
  m = warp_max(m);
  float s = 0.f;
  if (m != -INFINITY) {
    const float mk = __fmul_rn(m, k);
    if constexpr (kVec) {
      // four independent f32x2 accumulators, combined in a fixed order
      const f2 k2 = pk(k, k), nmk2 = pk(-mk, -mk);
      f2 acc[4] = {pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f), pk(0.f, 0.f)};
#pragma unroll
      for (int a = 0; a < kVecPerPass; ++a)
#pragma unroll
        for (int j = 0; j < N / 2; ++j)
          acc[(a * (N / 2) + j) & 3] = add2(acc[(a * (N / 2) + j) & 3], ex2x2(fma2(E::pair(t.v[a], j), k2, nmk2)));
      const float2 r = upk(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
      s = __fadd_rn(r.x, r.y);
    } else {
#pragma unroll
      for (int a = 0; a < kVecPerPass * N; ++a) s = __fadd_rn(s, ex2(fmaf(t.s[a], k, -mk)));
    }
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

// Statically sized shared state.
struct Fixed {
  float2 mass_warp[kWarps];
  float2 all_mass[kMaxCluster];       // (weight mass, p mass) of every block's chunk
  float pd[SPEC_MAX_GAMMA], qd[SPEC_MAX_GAMMA];
  float wsum[kMaxSlices][kWarps];     // owner: per-(slice, warp) weight sums
  int m, flags, owner, token, slice, warp_sel;
  float target_local, mass_out, run_sel;
};

// Dynamic shared memory, sized per launch (byte offsets).
struct Layout {
  int ring, vsw, vsp, all, wpart, local, rowM, rowInvS, rowArg, total;
};

__host__ __device__ inline Layout make_layout(int nslots, int cl, int slices) {
  Layout L;
  int off = 0;
  L.ring = off;
  L.vsw = off;                                          // phase B reuses the ring's space
  L.vsp = off + slices * kThreads * 4;
  const int need_a = kStages * kTileBytes, need_b = 2 * slices * kThreads * 4;
  off += need_a > need_b ? need_a : need_b;
  L.all = off;
  off += cl * nslots * 8;
  L.wpart = off;
  off += kWarps * nslots * 8;
  L.local = off;
  off += nslots * 8;
  L.rowM = off;
  off += nslots * 4;
  L.rowInvS = off;
  off += nslots * 4;
  L.rowArg = off;
  off += nslots * 4;
  L.total = (off + 15) & ~15;
  return L;
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------

template <class E, bool kVec, bool kMixed>
__global__ void __launch_bounds__(kThreads, 4) verify_kernel(const Args a) {
  using raw = typename E::raw;
  constexpr int N = E::kPerVec;
  constexpr int kPass = kThreads * kVecPerPass * N;     // elements per tile
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ Fixed fx;
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
  const int nslots = 2 * gmax + 1;                      // target rows 0..gmax, draft rows after
  const int qslot = gmax + 1;
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
  const int npass = hi > lo ? int((hi - lo + kPass - 1) / kPass) : 0;
  const int slices = npass * kVecPerPass;
  // the layout must be identical in every block of the cluster (blocks write into each
  // other's shared memory), so it is sized by the full chunk, not by this block's share
  const int slices_max = int((a.chunk + kPass - 1) / kPass) * kVecPerPass;
  const Layout L = make_layout(nslots, CL, slices_max);
  float2* all = reinterpret_cast<float2*>(dyn + L.all);
  float2* wpart = reinterpret_cast<float2*>(dyn + L.wpart);
  float2* local = reinterpret_cast<float2*>(dyn + L.local);
  float* rowM = reinterpret_cast<float*>(dyn + L.rowM);
  float* rowInvS = reinterpret_cast<float*>(dyn + L.rowInvS);
  int* rowArg = reinterpret_cast<int*>(dyn + L.rowArg);

  // Prefetch what the decision needs (draft ids, their logits, uniforms): lane i of warp 0
  // owns draft i; the loads complete while phase A streams.
  int d = -1;
  bool dvalid = false;
  float xp = 0.f, xq = 0.f, ua = 0.f;
  if (warp == 0 && lane < g) {
    d = a.draft_tokens[int64_t(b) * gmax + lane];
    dvalid = d >= 0 && int64_t(d) < V;
    if (sampling) {
      if (dvalid) {
        xp = E::at(P + int64_t(lane) * V, d);
        xq = E::at(Q + int64_t(lane) * V, d);
      }
      ua = a.u_accept[int64_t(b) * gmax + lane];
    }
  }

  // ---------------- phase A: one streaming pass over this block's chunk of every row -----
  // Row order: sampling [P_g, Q_{g-1}, P_{g-1}, ..., Q_0, P_0] (the rows a rejection most
  // often needs -- small m -- are read last); greedy [P_g, ..., P_0].
  const int nrows = sampling ? 2 * g + 1 : g + 1;
  auto row_of = [&](int r, int& slot) -> const raw* {
    if (!sampling || r == 0) {
      const int i = g - r;
      slot = i;
      return P + int64_t(i) * V;
    }
    const int i = g - 1 - ((r - 1) >> 1);
    if (r & 1) {
      slot = qslot + i;
      return Q + int64_t(i) * V;
    }
    slot = i;
    return P + int64_t(i) * V;
  };
  const int ntiles = nrows * npass;
  unsigned char* ring = dyn + L.ring;
  auto issue = [&](int t) {
    if constexpr (kVec) {
      if (t < ntiles) {
        const int r = t / npass, ps = t - r * npass;
        int slot;
        const raw* row = row_of(r, slot);
        const int64_t e0 = lo + int64_t(ps) * kPass;
        unsigned char* st = ring + (t % kStages) * kTileBytes;
#pragma unroll
        for (int q = 0; q < kVecPerPass; ++q) {
          const int64_t e = e0 + int64_t(q * kThreads + tid) * N;
          const bool in = e < hi;
          cp_async16(st + (q * kThreads + tid) * 16,
                     in ? static_cast<const void*>(row + e) : static_cast<const void*>(row), in ? 16 : 0);
        }
      }
      cp_async_commit();
    }
  };
  if constexpr (kVec) {
#pragma unroll
    for (int t = 0; t < kStages - 1; ++t) issue(t);
  }
  float rm = -INFINITY, rs = 0.f;   // running (max, sum) of a sampled row / argmax value
  int ri = INT_MAX;                 // running argmax id of a greedy row
  for (int t = 0; t < ntiles; ++t) {
    const int r = t / npass, ps = t - r * npass;
    int slot;
    const raw* row = row_of(r, slot);
    const int64_t e0 = lo + int64_t(ps) * kPass;
    Tile<E, kVec> tile;
    if constexpr (kVec) {
      issue(t + kStages - 1);
      cp_async_wait<kStages - 1>();
      const unsigned char* st = ring + (t % kStages) * kTileBytes;
#pragma unroll
      for (int q = 0; q < kVecPerPass; ++q)
        tile.v[q] = *reinterpret_cast<const uint4*>(st + (q * kThreads + tid) * 16);
      if (e0 + kPass > hi) {
        // partial tile: vectors q with e0 + (q*kThreads + tid)*N >= hi hold zero fill
        const int64_t left = hi - e0 - int64_t(tid) * N;
        const int nq = left <= 0 ? 0 : int((left + int64_t(kThreads) * N - 1) / (int64_t(kThreads) * N));
        tile.mask_tail(nq);
      }
    } else {
#pragma unroll
      for (int q = 0; q < kVecPerPass; ++q) {
        const int64_t e = e0 + int64_t(q * kThreads + tid) * N;
#pragma unroll
        for (int j = 0; j < N; ++j) tile.s[q * N + j] = (e + j < hi) ? E::at(row, e + j) : -INFINITY;
      }
    }
    if (sampling) tile_stats(tile, k, rm, rs);
    else tile_argmax(tile, e0, tid, rm, ri);
    if (ps == npass - 1) {
      if (!sampling) warp_argmax(rm, ri);
      if (lane == 0) wpart[warp * nslots + slot] = make_float2(rm, sampling ? rs : __int_as_float(ri));
      rm = -INFINITY;
      rs = 0.f;
      ri = INT_MAX;
    }
  }
  if constexpr (kVec) cp_async_wait<0>();
  if (npass == 0 && lane == 0) {
    // empty chunk: empty partials
    for (int r = 0; r < nrows; ++r) {
      int slot;
      row_of(r, slot);
      wpart[warp * nslots + slot] = make_float2(-INFINITY, sampling ? 0.f : __int_as_float(INT_MAX));
    }
  }
  __syncthreads();

  // block partial per row, warps merged in a fixed order
  for (int r = tid; r < nrows; r += kThreads) {
    int slot;
    row_of(r, slot);
    float2 acc = wpart[slot];
    for (int w = 1; w < kWarps; ++w) {
      const float2 p = wpart[w * nslots + slot];
      if (sampling) merge_ms(acc.x, acc.y, p.x, p.y, k);
      else if (better(p.x, __float_as_int(p.y), acc.x, __float_as_int(acc.y))) acc = p;
    }
    local[slot] = acc;
  }
  __syncthreads();

  // ---------------- exchange 1: push the partials into every block of the cluster --------
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (int idx = tid; idx < CL * nrows; idx += kThreads) {
    const int c = idx / nrows, r = idx - c * nrows;
    int slot;
    row_of(r, slot);
    float2* dst = cluster.map_shared_rank(&all[rank * nslots + slot], c);
    *dst = local[slot];
  }
  cluster.sync();

  // every block combines the C partials of each row in the same order -> identical results
  for (int r = tid; r < nrows; r += kThreads) {
    int slot;
    row_of(r, slot);
    if (sampling) {
      float M = -INFINITY;
      for (int c = 0; c < CL; ++c) M = fmaxf(M, all[c * nslots + slot].x);
      float S = 0.f;
      if (M != -INFINITY)
        for (int c = 0; c < CL; ++c) {
          const float2 p = all[c * nslots + slot];
          if (p.x != -INFINITY) S = __fadd_rn(S, __fmul_rn(p.y, ex2(__fmul_rn(p.x - M, k))));
        }
      rowM[slot] = M;
      rowInvS[slot] = __frcp_rn(S);
    } else {
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int c = 0; c < CL; ++c) {
        const float2 p = all[c * nslots + slot];
        if (better(p.x, __float_as_int(p.y), bv, bi)) { bv = p.x; bi = __float_as_int(p.y); }
      }
      rowArg[slot] = bi;
    }
  }
  __syncthreads();

  // ---------------- acceptance flags and the first rejection (warp 0) -----------------------
  if (warp == 0) {
    bool acc = false;
    if (lane < g) {
      if (sampling) {
        float p = NAN, q = NAN;
        if (dvalid) {
          p = prob(xp, k, __fmul_rn(rowM[lane], k), rowInvS[lane]);
          q = prob(xq, k, __fmul_rn(rowM[qslot + lane], k), rowInvS[qslot + lane]);
          // u < min(1, p/q): r = 0 when p = 0, r = +inf when q = 0 < p
          acc = (p == 0.f) ? (ua < 0.f) : (p >= q ? (ua < 1.f) : (__fmul_rn(ua, q) < p));
        }
        fx.pd[lane] = p;
        fx.qd[lane] = q;
      } else {
        acc = dvalid && d == rowArg[lane];
      }
    }
    const unsigned keep = __ballot_sync(kFull, acc);
    const unsigned rej = ~keep & (g >= 32 ? kFull : ((1u << g) - 1u));
    const int m = rej ? __ffs(rej) - 1 : g;
    const unsigned badmask = __ballot_sync(kFull, lane < g && !dvalid);
    if (lane == 0) {
      int f = flags;
      if (m < g && ((badmask >> m) & 1u)) f |= SPEC_ST_BAD_DRAFT;
      fx.m = m;
      fx.flags = f;
    }
  }
  __syncthreads();
  const int m = fx.m;

  if (!sampling) {
    if (rank == 0) {
      for (int i = tid; i <= gmax; i += kThreads) {
        int v = -1;
        if (i < m) v = a.draft_tokens[int64_t(b) * gmax + i];
        else if (i == m) v = rowArg[m];
        a.out_tokens[int64_t(b) * (gmax + 1) + i] = v;
      }
      if (a.diag)
        for (int i = tid; i < 2 * gmax + 1; i += kThreads) a.diag[int64_t(b) * (2 * gmax + 1) + i] = NAN;
      if (tid == 0) {
        a.num_accepted[b] = m;
        if (a.status) a.status[b] = fx.flags;
      }
    }
    return;
  }

  // ---------------- phase B: chunk mass of the distribution the last token is drawn from ---
  const bool pair = m < g;                 // rejection: residual of (p_m, q_m); else bonus p_g
  const raw* rp = P + int64_t(m) * V;
  const raw* rq = pair ? Q + int64_t(m) * V : nullptr;
  const float mkp = __fmul_rn(rowM[m], k), invp = rowInvS[m];
  const float mkq = pair ? __fmul_rn(rowM[qslot + m], k) : 0.f;
  const float invq = pair ? rowInvS[qslot + m] : 0.f;
  float* vsw = reinterpret_cast<float*>(dyn + L.vsw);   // per (slice, thread) weight sums
  float* vsp = reinterpret_cast<float*>(dyn + L.vsp);   // per (slice, thread) p sums
  // weights w (residual, or p on the bonus row) and p of one vector; elements past hi are 0
  auto vec_weights = [&](int64_t e, float (&w)[N], float (&p)[N]) {
    if constexpr (kVec) {
      if (e < hi) {
        const uint4 vp = ld_l2(rp + e);
        const f2 k2 = pk(k, k), nmkp = pk(-mkp, -mkp), ip = pk(invp, invp);
        if (pair) {
          const uint4 vq = ld_l2(rq + e);
          const f2 nmkq = pk(-mkq, -mkq), iq = pk(invq, invq);
#pragma unroll
          for (int j = 0; j < N / 2; ++j) {
            const float2 pp = upk(prob2(E::pair(vp, j), k2, nmkp, ip));
            const float2 qq = upk(prob2(E::pair(vq, j), k2, nmkq, iq));
            p[2 * j] = pp.x;
            p[2 * j + 1] = pp.y;
            w[2 * j] = residual(pp.x, qq.x);
            w[2 * j + 1] = residual(pp.y, qq.y);
          }
        } else {
#pragma unroll
          for (int j = 0; j < N / 2; ++j) {
            const float2 pp = upk(prob2(E::pair(vp, j), k2, nmkp, ip));
            p[2 * j] = w[2 * j] = pp.x;
            p[2 * j + 1] = w[2 * j + 1] = pp.y;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < N; ++j) w[j] = p[j] = 0.f;
      }
    } else {
#pragma unroll
      for (int j = 0; j < N; ++j) {
        if (e + j < hi) {
          p[j] = prob(E::at(rp, e + j), k, mkp, invp);
          w[j] = pair ? residual(p[j], prob(E::at(rq, e + j), k, mkq, invq)) : p[j];
        } else {
          w[j] = p[j] = 0.f;
        }
      }
    }
  };
  float wsum = 0.f, psum = 0.f;
  for (int ps = 0; ps < npass; ++ps) {
    const int64_t e0 = lo + int64_t(ps) * kPass;
#pragma unroll
    for (int q = 0; q < kVecPerPass; ++q) {
      float w[N], p[N];
      vec_weights(e0 + int64_t(q * kThreads + tid) * N, w, p);
      float sw = 0.f, sp = 0.f;
#pragma unroll
      for (int j = 0; j < N; ++j) {
        sw = __fadd_rn(sw, w[j]);
        sp = __fadd_rn(sp, p[j]);
      }
      const int s = ps * kVecPerPass + q;
      vsw[s * kThreads + tid] = sw;
      vsp[s * kThreads + tid] = sp;
      wsum = __fadd_rn(wsum, sw);
      psum = __fadd_rn(psum, sp);
    }
  }
  wsum = warp_sum(wsum);
  psum = warp_sum(psum);
  if (lane == 0) fx.mass_warp[warp] = make_float2(wsum, psum);
  __syncthreads();
  if (tid < CL) {
    float2 acc = fx.mass_warp[0];
    for (int w = 1; w < kWarps; ++w) {
      acc.x = __fadd_rn(acc.x, fx.mass_warp[w].x);
      acc.y = __fadd_rn(acc.y, fx.mass_warp[w].y);
    }
    float2* dst = cluster.map_shared_rank(&fx.all_mass[rank], tid);
    *dst = acc;
  }
  cluster.sync();

  // ---------------- which chunk holds u * total (every block, same order) ------------------
  if (tid == 0) {
    float R = 0.f, Pm = 0.f;
    for (int c = 0; c < CL; ++c) {
      R = __fadd_rn(R, fx.all_mass[c].x);
      Pm = __fadd_rn(Pm, fx.all_mass[c].y);
    }
    const bool use_w = !pair || R > 0.f;   // bonus: the weights are p itself
    int f = fx.flags;
    if (!use_w) f |= SPEC_ST_R_ZERO;
    const float total = use_w ? R : Pm;
    const float target = __fmul_rn(a.u_sample[b], total);
    int owner = -1, last = 0;
    float excl = 0.f, run = 0.f, excl_last = 0.f;
    for (int c = 0; c < CL; ++c) {
      const float w = use_w ? fx.all_mass[c].x : fx.all_mass[c].y;
      if (w > 0.f) { last = c; excl_last = run; }
      const float nr = __fadd_rn(run, w);
      if (owner < 0 && nr > target && w > 0.f) { owner = c; excl = run; }
      run = nr;
    }
    if (owner < 0) { owner = last; excl = excl_last; }
    fx.owner = owner;
    fx.flags = f | (use_w ? 0 : 0x100);   // 0x100: draw from p (internal)
    fx.target_local = __fsub_rn(target, excl);
    fx.mass_out = pair ? (use_w ? R : 0.f) : R;
  }
  __syncthreads();
  if (rank != fx.owner) return;

  // ---------------- owner block: locate the token from the per-vector sums -----------------
  const bool draw_p = !pair || (fx.flags & 0x100);
  const float* vs = draw_p ? vsp : vsw;
  const float tl = fx.target_local;
  // per-(slice, warp) sums; slice-major, warp-minor is ascending vocabulary order
  for (int s = 0; s < slices; ++s) {
    const float x = warp_sum(vs[s * kThreads + tid]);
    if (lane == 0) fx.wsum[s][warp] = x;
  }
  __syncthreads();
  if (tid == 0) {
    int ss = -1, sw = 0, ls = 0, lw = 0;
    float run = 0.f, base = 0.f, base_last = 0.f;
    for (int s = 0; s < slices && ss < 0; ++s)
      for (int w = 0; w < kWarps; ++w) {
        const float x = fx.wsum[s][w];
        if (x > 0.f) { ls = s; lw = w; base_last = run; }
        const float nr = __fadd_rn(run, x);
        if (nr > tl && x > 0.f) { ss = s; sw = w; base = run; break; }
        run = nr;
      }
    if (ss < 0) { ss = ls; sw = lw; base = base_last; }
    fx.slice = ss;
    fx.warp_sel = sw;
    fx.run_sel = base;
    fx.token = int(lo);
  }
  __syncthreads();
  if (warp == fx.warp_sel) {
    const int s = fx.slice;
    const float x = vs[s * kThreads + tid];
    float incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl = __fadd_rn(incl, y);
    }
    const float base = fx.run_sel;
    const unsigned hit = __ballot_sync(kFull, x > 0.f && __fadd_rn(base, incl) > tl);
    const unsigned pos = __ballot_sync(kFull, x > 0.f);
    const int sel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == sel) {
      const int ps = s / kVecPerPass, q = s - ps * kVecPerPass;
      const int64_t e = lo + int64_t(ps) * kPass + int64_t(q * kThreads + tid) * N;
      float w[N], p[N];
      vec_weights(e, w, p);
      float r = __fsub_rn(__fadd_rn(base, incl), x);
      int tok = -1, lastpos = -1;
#pragma unroll
      for (int j = 0; j < N; ++j) {
        const float wj = draw_p ? p[j] : w[j];
        r = __fadd_rn(r, wj);
        if (wj > 0.f) {
          lastpos = int(e) + j;
          if (tok < 0 && r > tl) tok = int(e) + j;
        }
      }
      fx.token = tok >= 0 ? tok : (lastpos >= 0 ? lastpos : int(lo));
    }
  }
  __syncthreads();

  const int tok = fx.token;
  for (int i = tid; i <= gmax; i += kThreads) {
    int v = -1;
    if (i < m) v = a.draft_tokens[int64_t(b) * gmax + i];
    else if (i == m) v = tok;
    a.out_tokens[int64_t(b) * (gmax + 1) + i] = v;
  }
  if (a.diag) {
    float* dg = a.diag + int64_t(b) * (2 * gmax + 1);
    for (int i = tid; i < gmax; i += kThreads) {
      dg[2 * i] = i < g ? fx.pd[i] : NAN;
      dg[2 * i + 1] = i < g ? fx.qd[i] : NAN;
    }
    if (tid == 0) dg[2 * gmax] = fx.mass_out;
  }
  if (tid == 0) {
    a.num_accepted[b] = m;
    if (a.status) a.status[b] = fx.flags & 0xff;
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

int slices_for(int64_t chunk, int dtype) {
  const int64_t per_pass = int64_t(kThreads) * kVecPerPass * (dtype == SPEC_BF16 ? 8 : 4);
  return int((chunk + per_pass - 1) / per_pass) * kVecPerPass;
}

std::mutex g_attr_mu;

template <class E, bool kVec, bool kMixed>
int launch(const Args& args, int B, int dtype, void* stream) {
  auto fn = verify_kernel<E, kVec, kMixed>;
  const Plan plan = make_plan(args.V);
  const int slices = slices_for(plan.chunk, dtype);
  if (slices > kMaxSlices) {
    set_error("V=%lld too large: %d vocabulary slices per block (max %d)", (long long)args.V, slices,
              kMaxSlices);
    return SPEC_ENOSPACE;
  }
  const Layout L = make_layout(2 * args.gmax + 1, plan.cl, slices);
  if (L.total > kMaxDynSmem) {
    set_error("shared memory plan of %d bytes exceeds %d", L.total, kMaxDynSmem);
    return SPEC_ENOSPACE;
  }
  if (int64_t(B) * plan.cl > INT_MAX) {
    set_error("B=%d too large for %d blocks per sequence", B, plan.cl);
    return SPEC_ENOSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  {
    // cluster sizes above 8 and dynamic shared memory above 48 KB need an opt-in; done once
    // per device and kernel
    static bool done[64] = {};
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(NonPortableClusterSizeAllowed)");
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)");
      if (dev < 64) done[dev] = true;
    }
  }
  Args a = args;
  a.chunk = plan.chunk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B * plan.cl), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = size_t(L.total);
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

template <bool kMixed>
int dispatch_on(const Args& a, int dtype, int B, void* stream) {
  const bool vec = vec_ok(a.target, dtype, a.V) && vec_ok(a.draft, dtype, a.V);
  if (dtype == SPEC_BF16)
    return vec ? launch<Bf16, true, kMixed>(a, B, dtype, stream) : launch<Bf16, false, kMixed>(a, B, dtype, stream);
  return vec ? launch<F32, true, kMixed>(a, B, dtype, stream) : launch<F32, false, kMixed>(a, B, dtype, stream);
}

}  // namespace
}  // namespace specverify

using namespace specverify;

extern "C" int spec_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens,
                                  const int32_t* num_draft, int B, int gmax, int V,
                                  int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                                  void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK || B == 0) return rc;
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
