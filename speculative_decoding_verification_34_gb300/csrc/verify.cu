// Greedy / sampling verification: one grid of independent blocks.
//
// What is computed follows the tutorial "投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡"
// (§3-§4 greedy verification and logit alignment, §7.1-§7.3 acceptance min(1,p/q), residual
// max(p-q,0)/R and the bonus draw) and the "M013" knowledge-base card (§03-§05, including the
// R = 0 remark).  How it is computed is this library's own design for sm_103a.
//
// Every row is cut into CL row chunks of `chunk` ids for the statistics pass and into DCL
// draw chunks of `dchunk` ids for the final draw.  The grid is a list of block-sized units
// in groups: group g holds the A units of sequence g, then the B units of sequence
// g - delta (delta groups ~ kDrawWaves waves of resident blocks).
//
//   A(b, row, c)  reads row chunk c of one row of sequence b once from HBM (128-bit loads),
//                 one ex2 per sampled element, and writes a (max, sum 2^((x-max)k)) partial, or
//                 an (argmax value, id) partial for greedy rows, to the workspace; the unit
//                 whose chunk holds the row's draft id also records that logit.  The last A
//                 unit of b to arrive (a counter) is the *decider*: it combines the partials in
//                 a fixed order, takes the acceptance decisions, finds m, and either writes the
//                 greedy result or publishes a plan for the final draw.
//   B(b, dc)      draws on the plan: draw chunk dc of the row the last token is drawn from --
//                 row m of p and q after a rejection, the bonus row otherwise; normally still
//                 in L2 -- reduced to its residual and p masses.  The last draw chunk of b to
//                 finish makes its block the *selector*: it locates the chunk holding u*R,
//                 rescans that chunk and writes the outputs.
//
// No block ever has to wait for another.  A B unit may wait a short, bounded while for its
// plan; each draw chunk then goes through a small state machine (untouched -> claimed by its B
// unit, or untouched -> given up -> taken by the decider) so that exactly one block processes
// it whatever the timing: the decider takes the chunks whose B units gave up before the plan
// was out, B units take the rest.  Every call returns the workspace's counters to zero.

#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace specverify {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
#ifndef SPEC_VEC_PER_PASS
#define SPEC_VEC_PER_PASS 4
#endif
constexpr int kVecPerPass = SPEC_VEC_PER_PASS;         // 16-byte vectors per thread per row pass
#ifndef SPEC_DRAW_VEC
#define SPEC_DRAW_VEC 4
#endif
#ifndef SPEC_PREFETCH
#define SPEC_PREFETCH 1
#endif
#ifndef SPEC_RING
#define SPEC_RING 0
#endif
constexpr int kDrawVec = SPEC_DRAW_VEC;                // vectors of each row per thread per draw step
constexpr bool kPrefetch = SPEC_PREFETCH != 0;         // row passes double-buffered in registers
constexpr int kRing = SPEC_RING;                       // >0: row passes staged through a ring of
                                                       // this many 16 KB shared-memory stages
constexpr int kStageBytes = kThreads * kVecPerPass * 16;   // one pass of one row (bf16 or fp32)
constexpr long long kMbarWaitNs = 2000000;             // bound on one stage wait (2 ms)
constexpr int kMaxChunks = 64;                         // row chunks, and draw chunks, per row
constexpr int kMaxSlices = 16;                         // kThreads-vector slices per draw chunk
#ifndef SPEC_CHUNK_TARGET
#define SPEC_CHUNK_TARGET 65536
#endif
#ifndef SPEC_DRAW_CHUNK_TARGET
#define SPEC_DRAW_CHUNK_TARGET 8192
#endif
#ifndef SPEC_DRAW_WAVES
#define SPEC_DRAW_WAVES 3.0
#endif
#ifndef SPEC_MIN_BLOCKS
#define SPEC_MIN_BLOCKS 4
#endif
constexpr int kChunkTarget = SPEC_CHUNK_TARGET;        // ids per row chunk before rounding
constexpr int kDrawChunkTarget = SPEC_DRAW_CHUNK_TARGET;   // ids per draw chunk before rounding
constexpr double kDrawWaves = SPEC_DRAW_WAVES;         // distance of the draw behind the rows
constexpr int kMinBlocks = SPEC_MIN_BLOCKS;            // resident blocks per SM the registers allow
constexpr int kMaxGroups = 65535;                      // grid z limit
constexpr int kPlanWaitIters = 32;                     // optional bounded wait of a B unit (~15 us)
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kInternalDrawP = 0x100;
// draw-chunk states (a chunk whose B unit saw the plan at once stays Free)
constexpr int kChunkFree = 0, kChunkMine = 1, kChunkGivenUp = 2, kChunkDecider = 3;

struct Args {
  const void* target;
  const void* draft;
  const int32_t* draft_tokens;
  const int32_t* num_draft;
  const float* temperature;
  const float* u_accept;
  const float* u_sample;
  int64_t V;
  int B;
  int gmax;
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* diag;
  int32_t* status;
};

struct Geo {
  int CL;       // row chunks per row
  int chunk;    // ids per row chunk (multiple of 8)
  int DCL;      // draw chunks per row
  int dchunk;   // ids per draw chunk (multiple of 8)
  int nslots;   // row slots per sequence: target rows 0..gmax, then draft rows 0..gmax-1
  int delta;    // B units of sequence b sit in group b + delta
  int b0, b1;   // sequences [b0, b1) of this launch
};

struct __align__(16) PlanRec {   // per sequence, published by the decider for the draw
  int m, g, flags, pair;
  float mkp, invp, mkq, invq;
};

// The published flag carries what a draw unit needs to start its loads: 0 = not yet, else
// bit 31 set, status flags in bits 20..27, pair in bit 16, m in bits 0..15.  The plan's
// normalisers are read from the record alongside the row loads.
__host__ __device__ inline int ready_word(const PlanRec& pr) {
  return int(0x80000000u | (unsigned(pr.flags & 0xff) << 20) | (unsigned(pr.pair & 1) << 16) | unsigned(pr.m & 0xffff));
}

struct Work {      // views into the caller's workspace
  int* cnt;        // [B] A arrivals               (counter header)
  int* bdone;      // [B] draw-chunk arrivals      (counter header)
  int* ready;      // [B] plan published           (counter header)
  int* state;      // [B][DCL] draw-chunk states   (counter header)
  PlanRec* plan;   // [B]
  float2* part;    // [B][nslots][CL]
  float* xd;       // [B][nslots] logit at the draft id of that row
  float2* mass;    // [B][DCL] (residual mass, p mass)
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
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
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
    const float v2 = __shfl_xor_sync(kFull, v, o);
    const int i2 = __shfl_xor_sync(kFull, i, o);
    if (better(v2, i2, v, i)) { v = v2; i = i2; }
  }
}

// p_v = 2^((x_v - M) k) / S, evaluated as ex2(x*k - M*k) * (1/S) with a rounded product.
__device__ __forceinline__ float prob(float x, float k, float mk, float inv_s) {
  return __fmul_rn(ex2(fmaf(x, k, -mk)), inv_s);
}

// max(p - q, 0) with a rounded difference: exactly 0 wherever p == q.
__device__ __forceinline__ float residual(float p, float q) { return fmaxf(__fsub_rn(p, q), 0.f); }

// Packed pairs of f32 (sm_100+ .f32x2 forms): each lane is rounded as the scalar fma.rn /
// add.rn would round it.  Only an explicit fma and sums of exponentials are packed: a packed
// product may be fused by the code generator into a following packed add or subtract.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 ex2x2(float2 a) { return make_float2(ex2(a.x), ex2(a.y)); }

// Element formats.  A 16-byte vector holds kPerVec elements.
struct Bf16 {
  using raw = uint16_t;
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kNegInf = 0xff80ff80u;   // two bf16 -inf
  __device__ __forceinline__ static float at(const raw* row, int64_t i) {
    return __uint_as_float(uint32_t(__ldg(row + i)) << 16);
  }
  __device__ __forceinline__ static float get(const uint4& v, int j) {
    const uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  // elements (2h, 2h+1) of a vector as a pair
  __device__ __forceinline__ static float2 pair(const uint4& v, int h) {
    const uint32_t w = h == 0 ? v.x : h == 1 ? v.y : h == 2 ? v.z : v.w;
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  // max over the vectors of one pass: bf16x2 max tree, one widening at the end
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
  static constexpr uint32_t kNegInf = 0xff800000u;
  __device__ __forceinline__ static float at(const raw* row, int64_t i) { return __ldg(row + i); }
  __device__ __forceinline__ static float get(const uint4& v, int j) {
    return __uint_as_float(j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w);
  }
  __device__ __forceinline__ static float2 pair(const uint4& v, int h) {
    return h == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ __forceinline__ static float tmax(const uint4 (&v)[kVecPerPass]) {
    float a = -INFINITY;
#pragma unroll
    for (int q = 0; q < kVecPerPass; ++q)
      a = fmaxf(a, fmaxf(fmaxf(__uint_as_float(v[q].x), __uint_as_float(v[q].y)),
                         fmaxf(__uint_as_float(v[q].z), __uint_as_float(v[q].w))));
    return a;
  }
};

// One pass of one row chunk: vector q of thread t covers ids e0 + (q*kThreads + t)*kPerVec
// .. + kPerVec - 1, coalesced across the block for every q.  Ids at or past hi read as -inf
// (vector path: whole vectors, since chunk ends are vector aligned there).
template <class E, bool kVec>
struct Tile {
  static constexpr int N = E::kPerVec;
  uint4 v[kVecPerPass];
  float s[kVec ? 1 : kVecPerPass * N];

  __device__ __forceinline__ void load(const typename E::raw* row, int64_t e0, int64_t hi, int tid) {
#pragma unroll
    for (int q = 0; q < kVecPerPass; ++q) {
      const int64_t e = e0 + int64_t(q * kThreads + tid) * N;
      if constexpr (kVec) {
        v[q] = e < hi ? ld_stream(row + e) : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
      } else {
#pragma unroll
        for (int j = 0; j < N; ++j) s[q * N + j] = (e + j < hi) ? E::at(row, e + j) : -INFINITY;
      }
    }
  }
  // a pass that lies entirely below hi: no bounds to check
  __device__ __forceinline__ void load_full(const typename E::raw* row, int64_t e0, int tid) {
    if constexpr (kVec) {
#pragma unroll
      for (int q = 0; q < kVecPerPass; ++q) v[q] = ld_stream(row + e0 + int64_t(q * kThreads + tid) * N);
    } else {
      load(row, e0, e0 + int64_t(kThreads) * kVecPerPass * N, tid);
    }
  }
  __device__ __forceinline__ float x(int q, int j) const {
    if constexpr (kVec) return E::get(v[q], j);
    else return s[q * N + j];
  }
  __device__ __forceinline__ float2 xp(int q, int h) const {
    if constexpr (kVec) return E::pair(v[q], h);
    else return make_float2(s[q * N + 2 * h], s[q * N + 2 * h + 1]);
  }
};

// Per-thread running (max m, sum of 2^((x-m)k)) over the passes of a chunk: the sum is rescaled
// when the max grows, and the warp is reduced once at the end (warp_stats).  Rows of -inf
// give (-inf, 0) without NaN.
template <class E, bool kVec>
__device__ __forceinline__ void thread_stats(const Tile<E, kVec>& t, float k, float& run_m, float& run_s) {
  constexpr int N = E::kPerVec;
  float m;
  if constexpr (kVec) {
    m = E::tmax(t.v);
  } else {
    m = -INFINITY;
#pragma unroll
    for (int a = 0; a < kVecPerPass * N; ++a) m = fmaxf(m, t.s[a]);
  }
  const float mn = fmaxf(run_m, m);
  const bool fin = mn != -INFINITY;
  const float mk = fin ? __fmul_rn(mn, k) : 0.f;
  const float scale = fin ? ex2(__fmul_rn(run_m - mn, k)) : 1.f;
  const float2 kk = make_float2(k, k), nmk = make_float2(-mk, -mk);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;   // four chains, combined in a fixed order
#pragma unroll
  for (int q = 0; q < kVecPerPass; ++q)
#pragma unroll
    for (int h = 0; h < N / 2; ++h) {
      const float2 e = ex2x2(fma2(t.xp(q, h), kk, nmk));
      if (h & 1) acc1 = add2(acc1, e);
      else acc0 = add2(acc0, e);
    }
  run_s = __fadd_rn(__fmul_rn(run_s, scale), __fadd_rn(__fadd_rn(acc0.x, acc0.y), __fadd_rn(acc1.x, acc1.y)));
  run_m = mn;
}

// the warp's (max, sum) from its threads' running statistics; every lane gets the result
__device__ __forceinline__ void warp_stats(float& m, float& s, float k) {
  const float M = warp_max(m);
  float S = 0.f;
  if (M != -INFINITY) S = warp_sum(m == -INFINITY ? 0.f : __fmul_rn(s, ex2(__fmul_rn(m - M, k))));
  m = M;
  s = S;
}

template <class E, bool kVec>
__device__ __forceinline__ void tile_argmax(const Tile<E, kVec>& t, int64_t e0, int tid, float& bv, int& bi) {
#pragma unroll
  for (int q = 0; q < kVecPerPass; ++q)
#pragma unroll
    for (int j = 0; j < E::kPerVec; ++j) {
      const int idx = int(e0 + int64_t(q * kThreads + tid) * E::kPerVec + j);
      const float v = t.x(q, j);
      if (better(v, idx, bv, bi)) { bv = v; bi = idx; }
    }
}

__device__ __forceinline__ int atom_cas(int* p, int cmp, int val) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.cas.b32 %0, [%1], %2, %3;" : "=r"(old) : "l"(p), "r"(cmp), "r"(val) : "memory");
  return old;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- bulk copies into shared memory, completed on an mbarrier -----------------------------

__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}
// one arrival that also announces `bytes` of transfer; the phase completes when they land
__device__ __forceinline__ void mbar_expect(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// waits for the phase of the given parity; false if kMbarWaitNs passed first
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = global_ns();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > kMbarWaitNs) return false;
  }
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)));
  return v;
}

// inclusive prefix sum over the warp's lanes, in a fixed association order
__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = int(threadIdx.x) & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v = __fadd_rn(v, y);
  }
  return v;
}

struct Shared {
  float2 wp[kWarps];
  float rowM[2 * SPEC_MAX_GAMMA + 1];
  float rowInvS[2 * SPEC_MAX_GAMMA + 1];
  int rowArg[SPEC_MAX_GAMMA + 1];
  float pd[SPEC_MAX_GAMMA], qd[SPEC_MAX_GAMMA];
  float wsum[kMaxSlices][kWarps];                 // selector: per-(slice, warp) weight sums
  int last, go, m, flags, owner, slice, warp_sel, token;
  unsigned taken[2];
  int err;
  float target_local, mass_out, run_sel;
  PlanRec plan;
  uint64_t bars[kRing > 0 ? kRing : 1];
};

// ------------------------------------------------------------------------------------------
// per-sequence context
// ------------------------------------------------------------------------------------------

template <class E, bool kMixed>
struct Seq {
  using raw = typename E::raw;
  int b, g, flags;
  bool sampling;
  float k;
  const raw* P;
  const raw* Q;

  __device__ __forceinline__ Seq(const Args& a, int b_) : b(b_) {
    g = a.num_draft ? __ldg(&a.num_draft[b]) : a.gmax;
    flags = 0;
    if (g < 0 || g > a.gmax) {
      g = g < 0 ? 0 : a.gmax;
      flags = SPEC_ST_CLAMPED_GAMMA;
    }
    float T = 0.f;
    if constexpr (kMixed) T = __ldg(&a.temperature[b]);
    sampling = kMixed && (T > 0.f);
    k = sampling ? kLog2e / T : 0.f;
    P = static_cast<const raw*>(a.target) + int64_t(b) * (a.gmax + 1) * a.V;
    Q = sampling ? static_cast<const raw*>(a.draft) + int64_t(b) * a.gmax * a.V : nullptr;
  }
  __device__ __forceinline__ bool slot_valid(int slot, int gmax) const {
    if (slot <= gmax) return slot <= g;
    return sampling && slot - gmax - 1 < g;
  }
  __device__ __forceinline__ int nrows() const { return sampling ? 2 * g + 1 : g + 1; }
  // r-th row read, in the order [P_g, Q_{g-1}, P_{g-1}, ..., Q_0, P_0] (sampling) or
  // [P_g, ..., P_0] (greedy)
  __device__ __forceinline__ int slot_of(int r, int gmax) const {
    if (!sampling || r == 0) return g - r;
    const int i = g - 1 - ((r - 1) >> 1);
    return (r & 1) ? gmax + 1 + i : i;
  }
  __device__ __forceinline__ const raw* row(int slot, int gmax, int64_t V) const {
    return slot <= gmax ? P + int64_t(slot) * V : Q + int64_t(slot - gmax - 1) * V;
  }
};

// weights of the N elements of one vector: w = residual (or p on the bonus row), and p
template <class E>
__device__ __forceinline__ void weights(const uint4& vp, const uint4& vq, bool pair, float k, float mkp, float invp,
                                        float mkq, float invq, float (&w)[E::kPerVec], float (&p)[E::kPerVec]) {
  // prob() and residual() with the exponent argument as a packed fma.  The products and the
  // difference stay scalar mul.rn / sub.rn, which are never fused: a product fused into the
  // difference would leave its rounding error behind where p == q must give exactly 0.
  const float2 kk = make_float2(k, k);
#pragma unroll
  for (int h = 0; h < E::kPerVec / 2; ++h) {
    const float2 ep = ex2x2(fma2(E::pair(vp, h), kk, make_float2(-mkp, -mkp)));
    p[2 * h] = __fmul_rn(ep.x, invp);
    p[2 * h + 1] = __fmul_rn(ep.y, invp);
    if (pair) {
      const float2 eq = ex2x2(fma2(E::pair(vq, h), kk, make_float2(-mkq, -mkq)));
      w[2 * h] = residual(p[2 * h], __fmul_rn(eq.x, invq));
      w[2 * h + 1] = residual(p[2 * h + 1], __fmul_rn(eq.y, invq));
    } else {
      w[2 * h] = p[2 * h];
      w[2 * h + 1] = p[2 * h + 1];
    }
  }
}

template <class E, bool kVec>
__device__ __forceinline__ uint4 vec_at(const typename E::raw* row, int64_t e, int64_t hi) {
  // one vector starting at id e; ids at or past hi read as -inf (prob() maps them to 0)
  if constexpr (kVec) {
    return e < hi ? ld_stream(row + e) : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
  } else {
    uint32_t u[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) u[h] = E::kNegInf;
    if constexpr (E::kPerVec == 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t x = (e + j < hi) ? uint32_t(__ldg(row + e + j)) : 0xff80u;
        u[j >> 1] = (j & 1) ? ((u[j >> 1] & 0x0000ffffu) | (x << 16)) : ((u[j >> 1] & 0xffff0000u) | x);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) u[j] = (e + j < hi) ? __float_as_uint(E::at(row, e + j)) : E::kNegInf;
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
}

// ------------------------------------------------------------------------------------------
// the draw: draw-chunk masses, then the selector
// ------------------------------------------------------------------------------------------

// Inverse CDF over the draw chunks of b: the owner chunk holds the smallest id whose running
// weight exceeds u * total; that chunk is rescanned in ascending id order.  Slice s of a draw
// chunk covers ids lo + s*kThreads*N .. + kThreads*N - 1, thread t the N ids from
// lo + (s*kThreads + t)*N, so (slice, warp, lane, element) is ascending id order.
template <class E, bool kVec, bool kMixed>
__device__ void select(const Args& a, const Geo& geo, const Work& w, const Seq<E, kMixed>& sq, const PlanRec pl,
                       Shared& sm) {
  using raw = typename E::raw;
  constexpr int N = E::kPerVec;
  constexpr int kSlice = kThreads * N;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int b = sq.b, gmax = a.gmax, DCL = geo.DCL;
  const bool pair = pl.pair != 0;
  if (warp == 0) {
    // chunk masses, lanes c and c + 32, prefix sums in ascending chunk order
    const float2* ms = w.mass + int64_t(b) * DCL;
    const float2 x0 = lane < DCL ? __ldcg(&ms[lane]) : make_float2(0.f, 0.f);
    const float2 x1 = lane + 32 < DCL ? __ldcg(&ms[lane + 32]) : make_float2(0.f, 0.f);
    const float r0 = warp_incl_scan(x0.x), p0 = warp_incl_scan(x0.y);
    const float rt0 = __shfl_sync(kFull, r0, 31), pt0 = __shfl_sync(kFull, p0, 31);
    const float r1 = __fadd_rn(rt0, warp_incl_scan(x1.x)), p1 = __fadd_rn(pt0, warp_incl_scan(x1.y));
    const float R = __shfl_sync(kFull, r1, 31), Pm = __shfl_sync(kFull, p1, 31);
    const bool use_w = !pair || R > 0.f;   // bonus: the weights are p itself
    const float w0 = use_w ? x0.x : x0.y, w1 = use_w ? x1.x : x1.y;
    const float i0 = use_w ? r0 : p0, i1 = use_w ? r1 : p1;
    const float total = use_w ? R : Pm;
    const float target = __fmul_rn(a.u_sample[b], total);
    // exclusive prefix of each chunk: the inclusive prefix of the one before it
    float e0 = __shfl_up_sync(kFull, i0, 1), e1 = __shfl_up_sync(kFull, i1, 1);
    const float t0 = __shfl_sync(kFull, i0, 31);
    if (lane == 0) { e0 = 0.f; e1 = t0; }
    const unsigned hit0 = __ballot_sync(kFull, w0 > 0.f && i0 > target);
    const unsigned hit1 = __ballot_sync(kFull, w1 > 0.f && i1 > target);
    const unsigned pos0 = __ballot_sync(kFull, w0 > 0.f), pos1 = __ballot_sync(kFull, w1 > 0.f);
    int owner;
    if (hit0) owner = __ffs(hit0) - 1;
    else if (hit1) owner = 32 + __ffs(hit1) - 1;
    else if (pos1) owner = 32 + 31 - __clz(pos1);   // rounding left u*total past the end
    else owner = pos0 ? 31 - __clz(pos0) : 0;
    const float excl = __shfl_sync(kFull, owner < 32 ? e0 : e1, owner & 31);
    if (lane == 0) {
      int f = pl.flags;
      if (!use_w) f |= SPEC_ST_R_ZERO | kInternalDrawP;
      sm.owner = owner;
      sm.flags = f;
      sm.target_local = __fsub_rn(target, excl);
      sm.mass_out = pair ? (use_w ? R : 0.f) : Pm;
    }
  }
  __syncthreads();
  const bool draw_p = !pair || (sm.flags & kInternalDrawP);
  const int64_t lo = int64_t(sm.owner) * geo.dchunk;
  const int64_t hi = lo + geo.dchunk < a.V ? lo + geo.dchunk : a.V;
  const raw* rp = sq.P + int64_t(pl.m) * a.V;
  const raw* rq = pair ? sq.Q + int64_t(pl.m) * a.V : rp;
  const int slices = int((hi - lo + kSlice - 1) / kSlice);
  for (int s = 0; s < slices; ++s) {
    const int64_t e = lo + int64_t(s) * kSlice + int64_t(tid) * N;
    float wv[N], pv[N];
    weights<E>(vec_at<E, kVec>(rp, e, hi), vec_at<E, kVec>(rq, e, pair ? hi : 0), pair, sq.k, pl.mkp, pl.invp, pl.mkq,
               pl.invq, wv, pv);
    float x = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) x = __fadd_rn(x, draw_p ? pv[j] : wv[j]);
    x = warp_sum(x);
    if (lane == 0) sm.wsum[s][warp] = x;
  }
  __syncthreads();
  const float tl = sm.target_local;
  if (tid == 0) {
    int ss = -1, sw = 0, ls = 0, lw = 0;
    float run = 0.f, base = 0.f, base_last = 0.f;
    for (int s = 0; s < slices && ss < 0; ++s)
      for (int wi = 0; wi < kWarps; ++wi) {
        const float x = sm.wsum[s][wi];
        if (x > 0.f) { ls = s; lw = wi; base_last = run; }
        const float nr = __fadd_rn(run, x);
        if (nr > tl && x > 0.f) { ss = s; sw = wi; base = run; break; }
        run = nr;
      }
    if (ss < 0) { ss = ls; sw = lw; base = base_last; }
    sm.slice = ss;
    sm.warp_sel = sw;
    sm.run_sel = base;
    sm.token = int(lo);
  }
  __syncthreads();
  if (warp == sm.warp_sel) {
    const int64_t e = lo + int64_t(sm.slice) * kSlice + int64_t(tid) * N;
    float wv[N], pv[N];
    weights<E>(vec_at<E, kVec>(rp, e, hi), vec_at<E, kVec>(rq, e, pair ? hi : 0), pair, sq.k, pl.mkp, pl.invp, pl.mkq,
               pl.invq, wv, pv);
    float x = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) x = __fadd_rn(x, draw_p ? pv[j] : wv[j]);
    const float incl = warp_incl_scan(x);
    const float base = sm.run_sel;
    const unsigned hit = __ballot_sync(kFull, x > 0.f && __fadd_rn(base, incl) > tl);
    const unsigned pos = __ballot_sync(kFull, x > 0.f);
    const int sel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == sel) {
      float r = __fsub_rn(__fadd_rn(base, incl), x);
      int tok = -1, lastpos = -1;
#pragma unroll
      for (int j = 0; j < N; ++j) {
        const float wj = draw_p ? pv[j] : wv[j];
        r = __fadd_rn(r, wj);
        if (wj > 0.f) {
          lastpos = int(e) + j;
          if (tok < 0 && r > tl) tok = int(e) + j;
        }
      }
      sm.token = tok >= 0 ? tok : (lastpos >= 0 ? lastpos : int(lo));
    }
  }
  __syncthreads();
  const int m = pl.m, tok = sm.token;
  for (int i = tid; i <= gmax; i += kThreads) {
    int v = -1;
    if (i < m) v = a.draft_tokens[int64_t(b) * gmax + i];
    else if (i == m) v = tok;
    a.out_tokens[int64_t(b) * (gmax + 1) + i] = v;
  }
  for (int c = tid; c < DCL; c += kThreads) w.state[int64_t(b) * DCL + c] = kChunkFree;
  if (tid == 0) {
    if (a.diag) a.diag[int64_t(b) * (2 * gmax + 1) + 2 * gmax] = sm.mass_out;
    a.num_accepted[b] = m;
    if (a.status) a.status[b] = sm.flags & 0xff;
    w.ready[b] = 0;
    w.bdone[b] = 0;
  }
  __syncthreads();
}

// one draw chunk: its residual and p masses; the last draw chunk of b to finish selects
template <class E, bool kVec, bool kMixed>
__device__ void draw_chunk(const Args& a, const Geo& geo, const Work& w, const Seq<E, kMixed>& sq, const PlanRec pl,
                           int dc, Shared& sm) {
  using raw = typename E::raw;
  constexpr int N = E::kPerVec;
  constexpr int kStep = kThreads * kDrawVec * N;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int b = sq.b;
  const bool pair = pl.pair != 0;
  const raw* rp = sq.P + int64_t(pl.m) * a.V;
  const raw* rq = pair ? sq.Q + int64_t(pl.m) * a.V : rp;
  const int64_t lo = int64_t(dc) * geo.dchunk;
  const int64_t hi = lo + geo.dchunk < a.V ? lo + geo.dchunk : a.V;
  float2 ws2 = make_float2(0.f, 0.f), ps2 = ws2;
  for (int64_t e0 = lo; e0 < hi; e0 += kStep) {
    uint4 vp[kDrawVec], vq[kDrawVec];
#pragma unroll
    for (int q = 0; q < kDrawVec; ++q) {
      const int64_t e = e0 + int64_t(q * kThreads + tid) * N;
      vp[q] = vec_at<E, kVec>(rp, e, hi);
      vq[q] = vec_at<E, kVec>(rq, e, pair ? hi : 0);
    }
#pragma unroll
    for (int q = 0; q < kDrawVec; ++q) {
      float wv[N], pv[N];
      weights<E>(vp[q], vq[q], pair, sq.k, pl.mkp, pl.invp, pl.mkq, pl.invq, wv, pv);
#pragma unroll
      for (int h = 0; h < N / 2; ++h) {
        ws2 = add2(ws2, make_float2(wv[2 * h], wv[2 * h + 1]));
        ps2 = add2(ps2, make_float2(pv[2 * h], pv[2 * h + 1]));
      }
    }
  }
  const float ws = warp_sum(__fadd_rn(ws2.x, ws2.y));
  const float ps = warp_sum(__fadd_rn(ps2.x, ps2.y));
  if (lane == 0) sm.wp[warp] = make_float2(ws, ps);
  __syncthreads();
  if (tid == 0) {
    float2 acc = sm.wp[0];
    for (int wi = 1; wi < kWarps; ++wi) {
      acc.x = __fadd_rn(acc.x, sm.wp[wi].x);
      acc.y = __fadd_rn(acc.y, sm.wp[wi].y);
    }
    if (!pair) acc.x = acc.y;
    w.mass[int64_t(b) * geo.DCL + dc] = acc;
    sm.last = atom_add_acq_rel(&w.bdone[b], 1) == geo.DCL - 1;
  }
  __syncthreads();
  if (sm.last) select<E, kVec, kMixed>(a, geo, w, sq, pl, sm);
}

// ------------------------------------------------------------------------------------------
// decider: combine the partials of sequence b, decide, then greedy result or the plan
// ------------------------------------------------------------------------------------------

// Entered by every thread of the block whose A unit arrived last, after the arrival atomic
// (acquire) and a block barrier: all partials and draft logits of b are visible.
template <class E, bool kVec, bool kMixed>
__device__ void decide(const Args& a, const Geo& geo, const Work& w, const Seq<E, kMixed>& sq, Shared& sm) {
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int b = sq.b, g = sq.g, gmax = a.gmax, CL = geo.CL;
  const float k = sq.k;
  // the per-draft inputs first: they do not depend on the combine below
  int d = -1;
  float u = 0.f, xp = 0.f, xq = 0.f;
  if (warp == 0 && lane < g) {
    d = __ldg(&a.draft_tokens[int64_t(b) * gmax + lane]);
    if (sq.sampling) {
      u = __ldg(&a.u_accept[int64_t(b) * gmax + lane]);
      xp = __ldcg(&w.xd[int64_t(b) * geo.nslots + lane]);
      xq = __ldcg(&w.xd[int64_t(b) * geo.nslots + gmax + 1 + lane]);
    }
  }
  // one warp per row: lanes take chunks c and c + 32 (at most 64 chunks)
  const float2* part = w.part + int64_t(b) * geo.nslots * CL;
  for (int slot = warp; slot < geo.nslots; slot += kWarps) {
    if (!sq.slot_valid(slot, gmax)) continue;
    const float2* pp = part + slot * CL;
    const float2 none = make_float2(-INFINITY, sq.sampling ? 0.f : __int_as_float(INT_MAX));
    const float2 p0 = lane < CL ? __ldcg(&pp[lane]) : none;
    const float2 p1 = lane + 32 < CL ? __ldcg(&pp[lane + 32]) : none;
    if (sq.sampling) {
      const float M = warp_max(fmaxf(p0.x, p1.x));
      float S = 0.f;
      if (M != -INFINITY) {
        const float t0 = p0.x == -INFINITY ? 0.f : __fmul_rn(p0.y, ex2(__fmul_rn(p0.x - M, k)));
        const float t1 = p1.x == -INFINITY ? 0.f : __fmul_rn(p1.y, ex2(__fmul_rn(p1.x - M, k)));
        S = warp_sum(__fadd_rn(t0, t1));
      }
      if (lane == 0) {
        sm.rowM[slot] = M;
        sm.rowInvS[slot] = __frcp_rn(S);
      }
    } else {
      float bv = p0.x;
      int bi = __float_as_int(p0.y);
      if (better(p1.x, __float_as_int(p1.y), bv, bi)) { bv = p1.x; bi = __float_as_int(p1.y); }
      warp_argmax(bv, bi);
      if (lane == 0) sm.rowArg[slot] = bi;
    }
  }
  if (tid < 2) sm.taken[tid] = 0u;
  __syncthreads();
  if (warp == 0) {
    bool acc = false;
    const bool valid = lane < g && d >= 0 && int64_t(d) < a.V;
    if (lane < g) {
      if (sq.sampling) {
        float p = NAN, q = NAN;
        if (valid) {
          const int qs = gmax + 1 + lane;
          p = prob(xp, k, __fmul_rn(sm.rowM[lane], k), sm.rowInvS[lane]);
          q = prob(xq, k, __fmul_rn(sm.rowM[qs], k), sm.rowInvS[qs]);
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
    const unsigned bad = __ballot_sync(kFull, lane < g && !valid);
    if (lane == 0) {
      int f = sq.flags;
      if (m < g && ((bad >> m) & 1u)) f |= SPEC_ST_BAD_DRAFT;
      sm.m = m;
      sm.flags = f;
    }
  }
  __syncthreads();
  const int m = sm.m;
  if (!sq.sampling) {
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
      w.cnt[b] = 0;
    }
    __syncthreads();
    return;
  }
  if (a.diag) {
    float* dg = a.diag + int64_t(b) * (2 * gmax + 1);
    for (int i = tid; i < gmax; i += kThreads) {
      dg[2 * i] = i < g ? sm.pd[i] : NAN;
      dg[2 * i + 1] = i < g ? sm.qd[i] : NAN;
    }
  }
  if (tid == 0) {
    PlanRec pr;
    pr.m = m;
    pr.g = g;
    pr.flags = sm.flags;
    pr.pair = m < g ? 1 : 0;
    pr.mkp = __fmul_rn(sm.rowM[m], k);
    pr.invp = sm.rowInvS[m];
    const int qs = gmax + 1 + m;
    pr.mkq = pr.pair ? __fmul_rn(sm.rowM[qs], k) : 0.f;
    pr.invq = pr.pair ? sm.rowInvS[qs] : 0.f;
    w.plan[b] = pr;
    sm.plan = pr;
    w.cnt[b] = 0;
    __threadfence();                 // the plan before the flag
    atomicExch(&w.ready[b], ready_word(pr));
    __threadfence();                 // the flag before the chunk states read below
  }
  __syncthreads();
  const PlanRec pl = sm.plan;
  // the draw chunks whose B units gave up before the plan was out are the decider's: with a
  // fence between the flag and these reads here, and between the give-up and the flag read in
  // the B unit, one of the two sides always sees the other
  if (tid < geo.DCL) {
    int* st = &w.state[int64_t(b) * geo.DCL + tid];
    __threadfence();
    if (ld_acquire(st) == kChunkGivenUp && atom_cas(st, kChunkGivenUp, kChunkDecider) == kChunkGivenUp)
      atomicOr(&sm.taken[tid >> 5], 1u << (tid & 31));
  }
  __syncthreads();
  const unsigned taken0 = sm.taken[0], taken1 = sm.taken[1];
  for (int c = 0; c < geo.DCL; ++c)
    if ((c < 32 ? taken0 >> c : taken1 >> (c - 32)) & 1u) draw_chunk<E, kVec, kMixed>(a, geo, w, sq, pl, c, sm);
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------

template <class E, bool kVec, bool kMixed>
__global__ void __launch_bounds__(kThreads, kMinBlocks) verify_kernel(const Args a, const Geo geo, const Work w) {
  using raw = typename E::raw;
  constexpr int N = E::kPerVec;
  constexpr int kPass = kThreads * kVecPerPass * N;
  __shared__ Shared sm;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  // blockIdx = (x, y, group).  y < nslots: the A unit of row slot y, row chunk x.  y >= nslots:
  // the B unit of draw chunk (y - nslots)*CL + x.  Blocks are dispatched in x-fastest order,
  // so a group's A units come first and its B units last.
  const int x = int(blockIdx.x), y = int(blockIdx.y), grp = geo.b0 + int(blockIdx.z);

  if (y < geo.nslots) {
    // ---------------- A unit: row chunk x of row slot y -------------------------------------
    const int b = grp, slot = y, c = x;
    if (b >= geo.b1) return;
    // The row's address does not depend on the sequence's num_draft and temperature: its
    // first two passes are started before those arrive.  A row past num_draft (or a draft
    // row of a greedy sequence) is inside the caller's tensors; its passes are dropped.
    const raw* row = slot <= a.gmax
                         ? static_cast<const raw*>(a.target) + (int64_t(b) * (a.gmax + 1) + slot) * a.V
                         : static_cast<const raw*>(a.draft) + (int64_t(b) * a.gmax + (slot - a.gmax - 1)) * a.V;
    const int64_t lo = int64_t(c) * geo.chunk;
    const int64_t hi = lo + geo.chunk < a.V ? lo + geo.chunk : a.V;
    auto fetch = [&](Tile<E, kVec>& t, int64_t e0) {
      if (e0 + kPass <= hi) t.load_full(row, e0, tid);
      else t.load(row, e0, hi, tid);
    };
    constexpr bool kRegs = kPrefetch && !(kRing > 0 && kVec);
    Tile<E, kVec> t0, t1;
    if constexpr (kRegs) {
      if (lo < hi) fetch(t0, lo);
      if (lo + kPass < hi) fetch(t1, lo + kPass);
    }
    const Seq<E, kMixed> sq(a, b);
    if (!sq.slot_valid(slot, a.gmax)) return;
    // the logit at this row's draft id, if it lies in this chunk: fetched once, up front
    const int i = slot <= a.gmax ? slot : slot - a.gmax - 1;
    bool has_d = false;
    float xv = 0.f;
    if (tid == 0 && sq.sampling && i < sq.g) {
      const int d = __ldg(&a.draft_tokens[int64_t(b) * a.gmax + i]);
      has_d = int64_t(d) >= lo && int64_t(d) < hi;
      if (has_d) xv = E::at(row, d);
    }
    float rm = -INFINITY, rs = 0.f;
    int ri = INT_MAX;
    auto consume = [&](const Tile<E, kVec>& t, int64_t e0) {
      if (sq.sampling) thread_stats(t, sq.k, rm, rs);
      else tile_argmax(t, e0, tid, rm, ri);
    };
    if constexpr (kRing > 0 && kVec) {
      // passes staged through a ring of kRing shared-memory stages by bulk copies: thread 0
      // keeps kRing passes in flight; a stage is refilled once every thread has its tile
      extern __shared__ __align__(128) unsigned char ring[];
      const int npass = lo < hi ? int((hi - lo + kPass - 1) / kPass) : 0;
      auto issue = [&](int p) {
        const int st = p % kRing;
        const int64_t e0 = lo + int64_t(p) * kPass;
        const int64_t n = hi - e0 < kPass ? hi - e0 : kPass;
        const unsigned bytes = unsigned(n * int64_t(sizeof(raw)));
        mbar_expect(&sm.bars[st], bytes);
        bulk_load(ring + st * kStageBytes, row + e0, bytes, &sm.bars[st]);
      };
      if (tid == 0) {
        sm.err = 0;
        for (int st = 0; st < kRing; ++st) mbar_init(&sm.bars[st]);
        mbar_fence_init();
        for (int p = 0; p < npass && p < kRing; ++p) issue(p);
      }
      __syncthreads();
      for (int p = 0; p < npass; ++p) {
        const int st = p % kRing;
        const int64_t e0 = lo + int64_t(p) * kPass;
        if (!mbar_wait(&sm.bars[st], unsigned(p / kRing) & 1u)) sm.err = 1;
        Tile<E, kVec> t;
#pragma unroll
        for (int q = 0; q < kVecPerPass; ++q) {
          const int off = q * kThreads + tid;
          t.v[q] = e0 + int64_t(off) * N < hi ? lds128(ring + st * kStageBytes + off * 16)
                                               : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
        }
        __syncthreads();
        if (tid == 0 && p + kRing < npass && !sm.err) issue(p + kRing);
        consume(t, e0);
      }
      if (sm.err) {
        // a stage wait ran out: wait, again bounded, for every copy this block issued, then
        // report the sequence
        if (tid == 0) {
          for (int p = npass - kRing > 0 ? npass - kRing : 0; p < npass; ++p)
            mbar_wait(&sm.bars[p % kRing], unsigned(p / kRing) & 1u);
          if (a.status) atomicOr(&a.status[b], SPEC_ST_TIMEOUT);
        }
        __syncthreads();
      }
    } else if constexpr (kRegs) {
      // two tiles in registers, both passes already in flight: each is refilled with the
      // pass after next as soon as it has been reduced
      for (int64_t e0 = lo; e0 < hi; e0 += 2 * kPass) {
        consume(t0, e0);
        if (e0 + 2 * kPass < hi) fetch(t0, e0 + 2 * kPass);
        if (e0 + kPass >= hi) break;
        consume(t1, e0 + kPass);
        if (e0 + 3 * kPass < hi) fetch(t1, e0 + 3 * kPass);
      }
    } else {
      for (int64_t e0 = lo; e0 < hi; e0 += kPass) {
        Tile<E, kVec> t;
        fetch(t, e0);
        consume(t, e0);
      }
    }
    if (sq.sampling) warp_stats(rm, rs, sq.k);
    else warp_argmax(rm, ri);
    if (lane == 0) sm.wp[warp] = make_float2(rm, sq.sampling ? rs : __int_as_float(ri));
    __syncthreads();
    if (warp == 0) {
      // the block's partial from the warps' partials, lanes in parallel
      float2 p = lane < kWarps ? sm.wp[lane] : make_float2(-INFINITY, sq.sampling ? 0.f : __int_as_float(INT_MAX));
      if (sq.sampling) {
        warp_stats(p.x, p.y, sq.k);
      } else {
        int pi = __float_as_int(p.y);
        warp_argmax(p.x, pi);
        p.y = __int_as_float(pi);
      }
      if (lane == 0) {
        if (has_d) w.xd[int64_t(b) * geo.nslots + slot] = xv;
        w.part[(int64_t(b) * geo.nslots + slot) * geo.CL + c] = p;
        // release: this thread's partial and draft logit before the count
        sm.last = atom_add_acq_rel(&w.cnt[b], 1) == geo.CL * sq.nrows() - 1;
      }
    }
    __syncthreads();
    if (sm.last) decide<E, kVec, kMixed>(a, geo, w, sq, sm);
    return;
  }

  if constexpr (kMixed) {
    // ---------------- B unit: draw chunk dc of sequence grp - delta -------------------------
    const int dc = (y - geo.nslots) * geo.CL + x;
    const int b = grp - geo.delta;
    if (dc >= geo.DCL || b < geo.b0 || b >= geo.b1) return;
    const Seq<E, kMixed> sq(a, b);
    // the plan flag is read while the sequence's metadata loads are still in flight
    int rdy = 0;
    if (tid == 0) rdy = ld_acquire(&w.ready[b]);
    if (!sq.sampling) return;
    if (tid == 0) {
      int* st = &w.state[int64_t(b) * geo.DCL + dc];
      // optional, bounded wait for the plan; correctness does not depend on it
      int it = 0, ns = 64;
      while (rdy == 0 && it < kPlanWaitIters) {
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;
        ++it;
        rdy = ld_acquire(&w.ready[b]);
      }
      bool mine = false;
      if (rdy != 0) {
        // the plan is out: the decider takes only given-up chunks, so this one stays ours
        // without a claim
        mine = true;
      } else if (atom_cas(st, kChunkFree, kChunkGivenUp) == kChunkFree) {
        // given up; if the plan appeared meanwhile, take the chunk back unless the decider has
        __threadfence();
        const int r2 = ld_acquire(&w.ready[b]);
        if (r2 != 0) {
          mine = atom_cas(st, kChunkGivenUp, kChunkMine) == kChunkGivenUp;
          rdy = r2;
        }
      }
      if (mine) {
        sm.plan.m = rdy & 0xffff;
        sm.plan.pair = (rdy >> 16) & 1;
        sm.plan.flags = (rdy >> 20) & 0xff;
        sm.plan.g = sq.g;
        // never fails for a well-formed workspace; keeps every read in bounds
        if (sm.plan.m > sq.g || (sm.plan.pair && sm.plan.m >= sq.g)) {
          mine = false;
          if (a.status) atomicOr(&a.status[b], SPEC_ST_TIMEOUT);
        }
      }
      sm.go = mine;
    }
    __syncthreads();
    if (!sm.go) return;
    // the normalisers, ordered after thread 0's acquire by the barrier; through L2 (an
    // earlier read of this line by the same SM may sit stale in L1).  Their load and the
    // rows' loads are in flight together.
    PlanRec pl = sm.plan;
    const float4 nf = __ldcg(reinterpret_cast<const float4*>(&w.plan[b]) + 1);
    pl.mkp = nf.x;
    pl.invp = nf.y;
    pl.mkq = nf.z;
    pl.invq = nf.w;
    draw_chunk<E, kVec, kMixed>(a, geo, w, sq, pl, dc, sm);
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

struct Split {
  int cl, chunk;     // row chunks
  int dcl, dchunk;   // draw chunks
};

void cut(int64_t V, int target, int& n, int& len) {
  int64_t c = (V + target - 1) / target;
  if (c < 1) c = 1;
  if (c > kMaxChunks) c = kMaxChunks;
  int64_t l = (V + c - 1) / c;
  l = (l + 7) / 8 * 8;
  n = int(c);
  len = int(l);
}

Split make_split(int64_t V) {
  Split s;
  cut(V, kChunkTarget, s.cl, s.chunk);
  cut(V, kDrawChunkTarget, s.dcl, s.dchunk);
  return s;
}

size_t align64(size_t x) { return (x + 63) & ~size_t(63); }

// Workspace layout.  The counters live in a header, the first eighth of the workspace (a
// function of workspace_bytes alone); the scratch lives after it.  Any call's scratch is
// therefore disjoint from any call's counters, whatever sizes successive calls use, and the
// counters (all zero between calls) stay valid.
struct WsLayout {
  size_t cnt, bdone, ready, state, plan, part, xd, mass, header, scratch_end;
};

size_t counter_bytes(int B, int64_t V) {
  const Split s = make_split(V);
  return 3 * align64(size_t(B) * 4) + align64(size_t(B) * s.dcl * 4);
}

size_t scratch_bytes(int B, int gmax, int64_t V) {
  const Split s = make_split(V);
  const size_t nslots = size_t(2 * gmax + 1);
  return align64(size_t(B) * sizeof(PlanRec)) + align64(size_t(B) * nslots * s.cl * 8) +
         align64(size_t(B) * nslots * 4) + align64(size_t(B) * s.dcl * 8);
}

size_t header_for(size_t ws_bytes) { return (ws_bytes / 8) & ~size_t(63); }

WsLayout ws_layout(int B, int gmax, int64_t V, size_t ws_bytes) {
  const Split s = make_split(V);
  const size_t nslots = size_t(2 * gmax + 1);
  WsLayout L;
  L.header = header_for(ws_bytes);
  L.cnt = 0;
  L.bdone = L.cnt + align64(size_t(B) * 4);
  L.ready = L.bdone + align64(size_t(B) * 4);
  L.state = L.ready + align64(size_t(B) * 4);
  size_t off = L.header;
  L.plan = off;
  off += align64(size_t(B) * sizeof(PlanRec));
  L.part = off;
  off += align64(size_t(B) * nslots * s.cl * 8);
  L.xd = off;
  off += align64(size_t(B) * nslots * 4);
  L.mass = off;
  off += align64(size_t(B) * s.dcl * 8);
  L.scratch_end = off;
  return L;
}

bool ws_fits(int B, int gmax, int64_t V, size_t ws_bytes) {
  return counter_bytes(B, V) <= header_for(ws_bytes) &&
         header_for(ws_bytes) + scratch_bytes(B, gmax, V) <= ws_bytes;
}

// smallest workspace (a multiple of 64 bytes) that fits a call of these sizes
size_t ws_required(int B, int gmax, int64_t V) {
  const size_t c = counter_bytes(B, V), sc = scratch_bytes(B, gmax, V);
  size_t w = align64(8 * (c + 64));
  const size_t w2 = align64((sc + 64) * 8 / 7 + 64);
  if (w2 > w) w = w2;
  while (!ws_fits(B, gmax, V, w)) w += 64;
  return w;
}

Work ws_views(void* ws, const WsLayout& L) {
  unsigned char* p = static_cast<unsigned char*>(ws);
  Work w;
  w.cnt = reinterpret_cast<int*>(p + L.cnt);
  w.bdone = reinterpret_cast<int*>(p + L.bdone);
  w.ready = reinterpret_cast<int*>(p + L.ready);
  w.state = reinterpret_cast<int*>(p + L.state);
  w.plan = reinterpret_cast<PlanRec*>(p + L.plan);
  w.part = reinterpret_cast<float2*>(p + L.part);
  w.xd = reinterpret_cast<float*>(p + L.xd);
  w.mass = reinterpret_cast<float2*>(p + L.mass);
  return w;
}

std::mutex g_occ_mu;

template <class E, bool kVec, bool kMixed>
int launch(const Args& args, int dtype, void* ws, size_t ws_bytes, void* stream) {
  auto fn = verify_kernel<E, kVec, kMixed>;
  const Split sp = make_split(args.V);
  const int64_t slice = int64_t(kThreads) * (dtype == SPEC_BF16 ? 8 : 4);
  const int64_t slices = (sp.dchunk + slice - 1) / slice;
  if (slices > kMaxSlices) {
    set_error("V=%lld too large: %lld slices per draw chunk (max %d)", (long long)args.V, (long long)slices,
              kMaxSlices);
    return SPEC_ENOSPACE;
  }
  // host-only checks first: nothing is enqueued when they fail
  if (!ws || !ws_fits(args.B, args.gmax, args.V, ws_bytes)) {
    set_error("workspace of %zu bytes is smaller than the %zu bytes needed", ws ? ws_bytes : size_t(0),
              ws_required(args.B, args.gmax, args.V));
    return SPEC_ENOSPACE;
  }
  if (reinterpret_cast<uintptr_t>(ws) % 64 != 0) {
    set_error("workspace must be 64-byte aligned");
    return SPEC_EINVAL;
  }
  const WsLayout L = ws_layout(args.B, args.gmax, args.V, ws_bytes);
  Geo geo;
  geo.CL = sp.cl;
  geo.chunk = sp.chunk;
  geo.DCL = sp.dcl;
  geo.dchunk = sp.dchunk;
  geo.nslots = kMixed ? 2 * args.gmax + 1 : args.gmax + 1;   // greedy-only reads no draft rows
  const int brows = kMixed ? (geo.DCL + geo.CL - 1) / geo.CL : 0;   // grid rows of B units
  const int G = geo.CL * (geo.nslots + brows);                       // units per group
  // B units of a sequence come about kDrawWaves waves of resident blocks after its A units
  // the shared-memory ring of the row passes (vector path only)
  const size_t dyn_smem = (kRing > 0 && kVec) ? size_t(kRing) * kStageBytes : 0;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  {
    static int cached[64] = {};
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (dev < 64 && cached[dev]) {
      per_sm = cached[dev];
    } else {
      if (dyn_smem > 0) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn_smem));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute (ring size)");
      }
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, dyn_smem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
      if (per_sm < 1) per_sm = 1;
      if (dev < 64) cached[dev] = per_sm;
    }
  }
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  const int64_t resident = int64_t(sms) * per_sm;
  geo.delta = kMixed ? int(std::ceil(kDrawWaves * double(resident) / double(G))) : 0;
  if (geo.delta > kMaxGroups / 2) geo.delta = kMaxGroups / 2;
  const Work w = ws_views(ws, L);
  // one launch covers at most kMaxGroups groups (the grid's z limit); larger batches take
  // several launches over consecutive sequence ranges, each complete on its own
  const int per_launch = kMaxGroups - geo.delta;
  for (int b0 = 0; b0 < args.B; b0 += per_launch) {
    geo.b0 = b0;
    geo.b1 = b0 + per_launch < args.B ? b0 + per_launch : args.B;
    const dim3 grid(unsigned(geo.CL), unsigned(geo.nslots + brows), unsigned(geo.b1 - b0 + geo.delta));
    fn<<<grid, kThreads, dyn_smem, static_cast<cudaStream_t>(stream)>>>(args, geo, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "verify kernel launch");
    count_launch();
  }
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
int dispatch_on(const Args& a, int dtype, void* ws, size_t ws_bytes, void* stream) {
  const bool vec = vec_ok(a.target, dtype, a.V) && vec_ok(a.draft, dtype, a.V);
  if (dtype == SPEC_BF16)
    return vec ? launch<Bf16, true, kMixed>(a, dtype, ws, ws_bytes, stream)
               : launch<Bf16, false, kMixed>(a, dtype, ws, ws_bytes, stream);
  return vec ? launch<F32, true, kMixed>(a, dtype, ws, ws_bytes, stream)
             : launch<F32, false, kMixed>(a, dtype, ws, ws_bytes, stream);
}

}  // namespace
}  // namespace specverify

using namespace specverify;

extern "C" size_t spec_verify_workspace_bytes(int B, int gmax, int V, int dtype) {
  if (B < 0 || gmax < 0 || gmax > SPEC_MAX_GAMMA || V < 1 || (dtype != SPEC_BF16 && dtype != SPEC_F32)) return 0;
  return ws_required(B, gmax, V);
}

extern "C" int spec_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens,
                                  const int32_t* num_draft, int B, int gmax, int V,
                                  int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK || B == 0) return rc;
  Args a = {};
  a.target = target_logits;
  a.draft_tokens = draft_tokens;
  a.num_draft = num_draft;
  a.V = V;
  a.B = B;
  a.gmax = gmax;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.status = status;
  return dispatch_on<false>(a, dtype, workspace, workspace_bytes, stream);
}

extern "C" int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                                  const int32_t* draft_tokens, const int32_t* num_draft,
                                  const float* temperature, const float* u_accept,
                                  const float* u_sample, int B, int gmax, int V,
                                  int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                  int32_t* status, void* workspace, size_t workspace_bytes,
                                  void* stream) {
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
  a.B = B;
  a.gmax = gmax;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.diag = diag;
  a.status = status;
  return dispatch_on<true>(a, dtype, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------------------------------
// spec_verify_sample_static: the same verification with a workspace compiled into the library
// ------------------------------------------------------------------------------------------
//
// For callers that cannot allocate device memory at the point of the call: a serving loop
// whose memory is fixed after start-up, or code between a framework's allocations that must
// not add one.  The workspace is one file-scope device array per device (every call of this
// entry point on that device shares it); its address is looked up once per device with
// cudaGetSymbolAddress.  Nothing is allocated, by this call or by any routine it calls.

namespace specverify {
namespace {

constexpr size_t kStaticWsBytes = SPEC_STATIC_WORKSPACE_BYTES;
static_assert(kStaticWsBytes % 64 == 0, "static workspace size");

// The shared workspace: its first eighth holds the counters, which must be zero before the
// first call and which every completed call leaves at zero; the scratch after it keeps the
// last call's values.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_mu;
void* g_static_ptr[64] = {};

// The device address of this device's array.  The first call on a device also clears the
// whole array and waits for that to finish.
int static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    set_error("device %d: the static workspace serves devices 0..63", dev);
    return SPEC_EINVAL;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static workspace");
    e = cudaMemset(p, 0, kStaticWsBytes);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static workspace");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static workspace");
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return SPEC_OK;
}

}  // namespace
}  // namespace specverify

extern "C" int spec_verify_sample_static(const void* target_logits, const void* draft_logits, int dtype,
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
  // sizes first, on the host: a call the array cannot hold touches nothing
  if (!ws_fits(B, gmax, V, kStaticWsBytes)) {
    set_error("B=%d gmax=%d V=%d needs a %zu-byte workspace; the static workspace holds %zu bytes "
              "(use spec_verify_sample with a caller-owned workspace)",
              B, gmax, V, ws_required(B, gmax, V), kStaticWsBytes);
    return SPEC_ENOSPACE;
  }
  void* ws = nullptr;
  rc = static_workspace(&ws);
  if (rc != SPEC_OK) return rc;
  Args a = {};
  a.target = target_logits;
  a.draft = draft_logits;
  a.draft_tokens = draft_tokens;
  a.num_draft = num_draft;
  a.temperature = temperature;
  a.u_accept = u_accept;
  a.u_sample = u_sample;
  a.V = V;
  a.B = B;
  a.gmax = gmax;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.diag = diag;
  a.status = status;
  return dispatch_on<true>(a, dtype, ws, kStaticWsBytes, stream);
}

extern "C" int spec_verify_plan(int V, int dtype, int* ctas_per_seq, int* chunk) {
  clear_error();
  if (V < 1 || (dtype != SPEC_BF16 && dtype != SPEC_F32) || !ctas_per_seq || !chunk) {
    set_error("bad arguments to spec_verify_plan");
    return SPEC_EINVAL;
  }
  const Split p = make_split(V);
  *ctas_per_seq = p.cl;
  *chunk = p.chunk;
  return SPEC_OK;
}
