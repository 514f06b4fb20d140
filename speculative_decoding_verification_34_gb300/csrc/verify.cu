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
//                 whose chunk holds the row's draft id also records that logit.  Each A unit
//                 counts its arrival when it starts reading; the last of b to arrive is the
//                 *decider*: once its own row is done it combines the partials in a fixed
//                 order, takes the acceptance decisions, finds m, and either writes the greedy
//                 result or publishes a plan for the final draw.
//   B(b, dc)      draws on the plan: draw chunk dc of the row the last token is drawn from --
//                 row m of p and q after a rejection, the bonus row otherwise; normally still
//                 in L2 -- reduced to its residual and p masses.  Each draw chunk counts its
//                 arrival as it starts; the last of b to arrive makes its block the
//                 *selector*: it locates the chunk holding u*R, rescans that chunk and writes
//                 the outputs.
//
// No block waits for a block that has not started.  The decider waits, bounded, for the
// partials of the A units of its sequence that arrived before it, the selector for the masses
// of the draw chunks that arrived before it (they are running); a B unit
// may wait a short, bounded while for its plan, then gives up; each draw chunk then goes through a small state machine (untouched -> claimed by its B
// unit, or untouched -> given up -> taken by the decider) so that exactly one block processes
// it whatever the timing: the decider takes the chunks whose B units gave up before the plan
// was out, B units take the rest.  Every call returns the workspace's counters to zero.

#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "schedule.h"

namespace specverify {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerPass = 4;                 // 16-byte vectors per thread per row pass
constexpr int kDrawVec = 4;                    // vectors of each row per thread per draw step
constexpr long long kWaitNs = 2000000;         // bound on any wait for another block (2 ms)
constexpr int kMaxChunks = 64;                 // row chunks per row
constexpr int kMaxDrawChunks = 16;             // draw chunks per row
constexpr int kSubPerLane = kMaxDrawChunks * kWarps / 32;   // selector: sub-ranges per lane
constexpr int kPartBuf = 512;                  // decider: row partials staged in shared memory at once
static_assert(kPartBuf % kThreads == 0 && kMaxChunks < kPartBuf, "partial batches");
static_assert(SPEC_MAX_GAMMA < kThreads, "one output per thread");
constexpr int kChunkTarget = 65536;            // ids per row chunk before rounding
constexpr int kDrawChunkTarget = 16384;        // ids per draw chunk before rounding
constexpr double kDrawWaves = 1.5;             // distance of the draw behind the rows
constexpr long long kDeferBytes = 32LL << 20;  // draw rows deferred to the end of a call
constexpr int kMinBlocks = 4;                  // resident blocks per SM the registers allow
constexpr int kMaxGroups = 65535;                      // grid z limit
constexpr int kPlanWaitIters = 64;                     // optional bounded wait of a B unit (~31 us)
constexpr unsigned kFull = 0xffffffffu;
// target rows per sequence the greedy kernel handles: a chain's gmax+1, a tree's nmax+1
constexpr int kMaxRows = (SPEC_MAX_TREE_NODES > SPEC_MAX_GAMMA ? SPEC_MAX_TREE_NODES : SPEC_MAX_GAMMA) + 1;
constexpr float kLog2e = 1.4426950408889634f;
// draw-chunk states (a chunk whose B unit saw the plan at once stays Free)
constexpr int kChunkFree = 0, kChunkMine = 1, kChunkGivenUp = 2, kChunkDecider = 3;

struct Args {
  const void* saved;    // split layout: target row 0 of every sequence, [B][V]; else null
  const void* target;   // [B][gmax+1][V], or rows 1..gmax as [B][gmax][V] in the split layout
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
  const int32_t* parents;   // tree verification: node parents [B][gmax]; else null
  int32_t* path_nodes;      // tree verification: accepted path [B][gmax]
  // the commit of the same round, done by the thread that writes the sequence's outputs
  // (kv_target null: no commit)
  int32_t* kv_target;       // [B] t, read and written
  int32_t* kv_draft;        // [B] or null
  int kv_add;               // 1 when the correction/bonus token counts as processed
  int32_t* history;         // [B][cap] or null
  int32_t* committed_len;   // [B] (with history)
  int cap;
};

struct Geo {
  int CL;       // row chunks per row
  int chunk;    // ids per row chunk (multiple of 8)
  int DCL;      // draw chunks per row
  int dchunk;   // ids per draw chunk (multiple of 8)
  int nslots;   // row slots per sequence: target rows 0..gmax, then draft rows 0..gmax-1
  int delta;    // B units of sequence b sit in group b + delta (see draw_group_seq)
  int ndefer;   // the first ndefer sequences of a launch draw after all of its row units
  int b0, b1;   // sequences [b0, b1) of this launch
};

struct __align__(16) PlanRec {   // per sequence, published by the decider for the draw
  int m, g, flags, pair;
  float mkp, invp, mkq, invq;
  float taup, tauq;   // truncated sampling: the smallest kept logit of row m of p and of q
};

// The published flag carries what a draw unit needs to start its loads: 0 = not yet, else
// bit 31 set, status flags in bits 20..27, pair in bit 16, m in bits 0..15.  The plan's
// normalisers are read from the record alongside the row loads.
__host__ __device__ inline int ready_word(const PlanRec& pr) {
  return int(0x80000000u | (unsigned(pr.flags & 0xff) << 20) | (unsigned(pr.pair & 1) << 16) | unsigned(pr.m & 0xffff));
}

struct Work {      // views into the caller's workspace: every word is 0 between calls
  int* cnt;        // [B] A arrivals
  int* bdone;      // [B] draw-chunk arrivals
  uint64_t* planw; // [B][4] published plan words
  int* state;      // [B][DCL] draw-chunk states
  uint64_t* part;  // [B][nslots][CL] published row partials (0 while unwritten)
  uint64_t* xd;    // [B][nslots] published logit at the draft id of that row
  uint64_t* mass;  // [B][DCL][kWarps] published sub-range masses (residual, -p)
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

// 64-bit relaxed accesses at GPU scope: single-copy atomic, so a reader sees either the old
// word or the whole new one.  A row unit publishes its partial this way, with no fence: the
// word is nonzero by construction and the slot is zero until written, so the reader polls the
// slot itself instead of relying on the order of the partial and the arrival count.
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int atom_add_relaxed(int* p, int v) {
  int old;
  asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
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

// Published words.  A row partial is (M bits | S bits << 32) for sampling rows -- S >= 1 when M
// is finite and M = -inf when S = 0, so the word is never 0 -- and (value bits | ~id << 32)
// for greedy rows (~id != 0).  The logit at a draft id is (bits | 1 << 32).  NaN values are
// stored as the canonical quiet NaN.
__device__ __forceinline__ uint32_t canon_bits(float x) { return x != x ? 0x7fc00000u : __float_as_uint(x); }
__device__ __forceinline__ uint64_t pack_word(uint32_t lo, uint32_t hi) { return uint64_t(lo) | (uint64_t(hi) << 32); }

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

// the warp's (max, sum) from its threads' running statistics; every lane gets the result.  A
// part whose max is -inf holds no finite logit: its sum is 0, or NaN when it met a NaN logit,
// and is carried as it is, so that a NaN anywhere in a row reaches the row's sum.
__device__ __forceinline__ void warp_stats(float& m, float& s, float k) {
  const float M = warp_max(m);
  const float S = warp_sum(m == -INFINITY ? s : __fmul_rn(s, ex2(__fmul_rn(m - M, k))));
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

// The greedy-only kernel's cheaper form of the same running argmax (vector path).  A thread's
// ids ascend with the pass, then q, then j, so a later element wins only with a strictly larger
// value: per pass the tile's max comes from a packed max tree, and the whole tile is kept in
// registers when that max beats the running one.  Once the chunk is done the kept tile is
// searched for the first element holding the max.  A tile of NaN only is never kept.
template <class E>
struct KeptTile {
  float m = -INFINITY;
  int64_t e0 = -1;
  uint4 v[kVecPerPass];

  __device__ __forceinline__ void offer(const Tile<E, true>& t, int64_t te0) {
    const float tm = E::tmax(t.v);
    if (tm > m || (e0 < 0 && tm == tm)) {
      m = tm;
      e0 = te0;
#pragma unroll
      for (int q = 0; q < kVecPerPass; ++q) v[q] = t.v[q];
    }
  }
  __device__ __forceinline__ void settle(int tid, float& bv, int& bi) const {
    if (e0 < 0) return;
    int found = INT_MAX;
#pragma unroll
    for (int q = 0; q < kVecPerPass; ++q)
#pragma unroll
      for (int j = 0; j < E::kPerVec; ++j)
        if (found == INT_MAX && E::get(v[q], j) == m) found = int(e0 + int64_t(q * kThreads + tid) * E::kPerVec + j);
    bv = m;
    bi = found;
  }
};

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

__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
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
  int rowArg[kMaxRows];
  int tpar[kMaxRows], ttok[kMaxRows], tpath[kMaxRows];   // tree verification
  unsigned char tacc[kMaxRows], tdep[kMaxRows];
  int tbest;
  float pd[SPEC_MAX_GAMMA], qd[SPEC_MAX_GAMMA];
  int last, go, m, flags, flags_extra, owner, token, lastpos;
  unsigned taken[2];
  int err;
  float base, target, mass_out;
  int hist;                 // history slot of the round's first token, -1: no history write
  PlanRec plan;
  float2 pbuf[kPartBuf];    // decider: one batch of rows' partials
};

// ------------------------------------------------------------------------------------------
// per-sequence context
// ------------------------------------------------------------------------------------------

// Target row i of sequence b.  In the split layout row 0 (the prediction saved from the last
// round) has an array of its own and rows 1..gmax are contiguous per sequence.
template <class E>
__device__ __forceinline__ const typename E::raw* target_row(const Args& a, int b, int i) {
  using raw = typename E::raw;
  if (a.saved) {
    return i == 0 ? static_cast<const raw*>(a.saved) + int64_t(b) * a.V
                  : static_cast<const raw*>(a.target) + (int64_t(b) * a.gmax + (i - 1)) * a.V;
  }
  return static_cast<const raw*>(a.target) + (int64_t(b) * (a.gmax + 1) + i) * a.V;
}

template <class E, bool kMixed>
struct Seq {
  using raw = typename E::raw;
  int b, g, flags;
  bool sampling;
  float k;
  const raw* P0;   // target row 0
  const raw* P1;   // target row 1; rows i >= 1 follow it V apart
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
    P0 = target_row<E>(a, b, 0);
    P1 = target_row<E>(a, b, 1);
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
  __device__ __forceinline__ const raw* prow(int i, int64_t V) const { return i == 0 ? P0 : P1 + int64_t(i - 1) * V; }
};

// weights of the N elements of one vector: w = residual (or p on the bonus row), and p.
// kTrunc: ids whose logit is below the row's kept threshold (taup, tauq) have probability 0.
template <class E, bool kTrunc = false>
__device__ __forceinline__ void weights(const uint4& vp, const uint4& vq, bool pair, float k, float mkp, float invp,
                                        float mkq, float invq, float (&w)[E::kPerVec], float (&p)[E::kPerVec],
                                        float taup = 0.f, float tauq = 0.f) {
  // prob() and residual() with the exponent argument as a packed fma.  The products and the
  // difference stay scalar mul.rn / sub.rn, which are never fused: a product fused into the
  // difference would leave its rounding error behind where p == q must give exactly 0.
  const float2 kk = make_float2(k, k);
#pragma unroll
  for (int h = 0; h < E::kPerVec / 2; ++h) {
    const float2 xp = E::pair(vp, h);
    const float2 ep = ex2x2(fma2(xp, kk, make_float2(-mkp, -mkp)));
    p[2 * h] = __fmul_rn(ep.x, invp);
    p[2 * h + 1] = __fmul_rn(ep.y, invp);
    if constexpr (kTrunc) {
      if (!(xp.x >= taup)) p[2 * h] = 0.f;
      if (!(xp.y >= taup)) p[2 * h + 1] = 0.f;
    }
    if (pair) {
      const float2 xq = E::pair(vq, h);
      const float2 eq = ex2x2(fma2(xq, kk, make_float2(-mkq, -mkq)));
      float q0 = __fmul_rn(eq.x, invq), q1 = __fmul_rn(eq.y, invq);
      if constexpr (kTrunc) {
        if (!(xq.x >= tauq)) q0 = 0.f;
        if (!(xq.y >= tauq)) q1 = 0.f;
      }
      w[2 * h] = residual(p[2 * h], q0);
      w[2 * h + 1] = residual(p[2 * h + 1], q1);
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

// The published word at p, given a first read v of it: once it is there (its writer has counted
// its arrival, which this block has seen, so it is running and stores the word when its part
// is done), the slot returns to zero for the next call.  Bounded: after kWaitNs the sequence is
// flagged SPEC_ST_TIMEOUT and 0 is used.
// First reads of several words are issued together, then settled one by one.
__device__ __forceinline__ uint64_t settle_word(uint64_t* p, uint64_t v, Shared& sm) {
  if (v == 0) {
    const long long t0 = global_ns();
    while ((v = ld_relaxed_u64(p)) == 0)
      if (global_ns() - t0 > kWaitNs) {
        atomicOr(&sm.flags_extra, SPEC_ST_TIMEOUT);
        break;
      }
  }
  *p = 0;
  return v;
}

// The commit of sequence b's round (tutorial §5.1-§5.2; card §06), when the call carries one:
// the caches are trimmed to t + m and hold t + m + 1 once the last token has been fed; the m + 1
// emitted tokens (the drafts d_0..d_{m-1}, then the last token) are appended to the history at
// committed_len, or, if they would pass its capacity, the sequence is left untouched.  The
// current lengths are loaded when the thread that commits starts its part of the round
// (commit_load), so that no load trails the outputs.
struct CommitIn {
  int kvt, kvd, clen;
};

__device__ __forceinline__ CommitIn commit_load(const Args& a, int b) {
  CommitIn c = {0, 0, 0};
  if (!a.kv_target) return c;
  c.kvt = a.kv_target[b];
  if (a.kv_draft) c.kvd = a.kv_draft[b];
  if (a.history) c.clen = a.committed_len[b];
  return c;
}

// Writes the new lengths; returns the status bits to add and, in *hist, the history slot the
// m + 1 tokens go to (-1: none), which the output threads fill.  Called by one thread.
__device__ __forceinline__ int commit_apply(const Args& a, int b, int m, const CommitIn& c, int* hist) {
  *hist = -1;
  if (!a.kv_target) return 0;
  const int n = m + 1;
  if (a.history) {
    if (c.clen < 0 || c.clen > a.cap - n) return SPEC_ST_HISTORY_FULL;
    *hist = c.clen;
    a.committed_len[b] = c.clen + n;
  }
  a.kv_target[b] = c.kvt + m + a.kv_add;
  if (a.kv_draft) a.kv_draft[b] = c.kvd + m + a.kv_add;
  return 0;
}

// Output i of sequence b (i = 0..gmax): token v, and its history copy when the commit has one.
__device__ __forceinline__ void put_output(const Args& a, int b, int i, int m, int v, int hist) {
  a.out_tokens[int64_t(b) * (a.gmax + 1) + i] = v;
  if (hist >= 0 && i <= m) a.history[int64_t(b) * a.cap + hist + i] = v;
}

// ------------------------------------------------------------------------------------------
// the draw: per-warp masses of each draw chunk, then the selector
// ------------------------------------------------------------------------------------------
//
// Draw chunk dc covers ids [dc*dchunk, (dc+1)*dchunk); warp w of the unit that reduces it owns
// the contiguous sub-range [dc*dchunk + w*wlen, + wlen) with wlen = dchunk / kWarps, a whole
// number of vectors.  Sub-range j = dc*kWarps + w is therefore the j-th slice of the row in
// ascending id order, and its (residual, p) masses sit at mass[b][j].  In a warp step, vector
// q of lane l covers the ids e0 + (q*32 + l)*N .. + N-1, so (step, q, lane, element) is
// ascending id order too.

// Inverse CDF over the sub-range masses of b: warp 0 finds the owner sub-range (the one
// holding the smallest id whose running weight exceeds u * total), then the block rescans it
// in ascending id order, one 16-byte vector of p (and q) per thread per step.  Called by every
// thread of the block.
template <class E, bool kVec, bool kMixed, bool kTrunc = false>
__device__ void select(const Args& a, const Geo& geo, const Work& w, const Seq<E, kMixed>& sq, const PlanRec pl,
                       Shared& sm) {
  using raw = typename E::raw;
  constexpr int N = E::kPerVec;
  constexpr int kStep = kThreads * N;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int b = sq.b, gmax = a.gmax;
  const bool pair = pl.pair != 0;
  // what the outputs and the commit need besides the token, loaded before the masses so that
  // no round trip trails the draw: u, the accepted drafts (thread i holds d_i) and the lengths
  const float us = warp == 0 ? __ldg(&a.u_sample[b]) : 0.f;
  const int dtok = tid < pl.m ? __ldg(&a.draft_tokens[int64_t(b) * gmax + tid]) : -1;
  const CommitIn cin = tid == 0 ? commit_load(a, b) : CommitIn{0, 0, 0};
  if (tid == 0) sm.flags_extra = 0;
  __syncthreads();
  if (warp == 0) {
    const int nsub = geo.DCL * kWarps;
    const int per = (nsub + 31) / 32;   // consecutive sub-ranges per lane (at most kSubPerLane)
    uint64_t* ms = w.mass + int64_t(b) * nsub;
    uint64_t raw_w[kSubPerLane];
#pragma unroll
    for (int i = 0; i < kSubPerLane; ++i) {
      const int j = lane * per + i;
      raw_w[i] = (i < per && j < nsub) ? ld_relaxed_u64(&ms[j]) : 0;
    }
    float2 x[kSubPerLane];
    float lr = 0.f, lp = 0.f;
#pragma unroll
    for (int i = 0; i < kSubPerLane; ++i) {
      const int j = lane * per + i;
      x[i] = make_float2(0.f, 0.f);
      if (i < per && j < nsub) {
        const uint64_t v = settle_word(&ms[j], raw_w[i], sm);
        x[i] = make_float2(__uint_as_float(uint32_t(v)), -__uint_as_float(uint32_t(v >> 32)));
      }
      lr = __fadd_rn(lr, x[i].x);
      lp = __fadd_rn(lp, x[i].y);
    }
    const float ir = warp_incl_scan(lr), ip = warp_incl_scan(lp);
    const float R = __shfl_sync(kFull, ir, 31), Pm = __shfl_sync(kFull, ip, 31);
    const bool use_w = !pair || R > 0.f;   // bonus: the weights are p itself
    const float total = use_w ? R : Pm;
    const float target = __fmul_rn(us, total);
    const float incl = use_w ? ir : ip, mine = use_w ? lr : lp;
    float excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = 0.f;
    // owner lane: the first whose running total passes the target (else the last with weight)
    const unsigned hit = __ballot_sync(kFull, mine > 0.f && incl > target);
    const unsigned pos = __ballot_sync(kFull, mine > 0.f);
    const int ol = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == ol) {
      float run = excl, base = excl, base_last = excl;
      int found = -1, lastj = 0;
#pragma unroll
      for (int i = 0; i < kSubPerLane; ++i) {
        if (i >= per || found >= 0) continue;
        const float wv = use_w ? x[i].x : x[i].y;
        const float nr = __fadd_rn(run, wv);
        if (wv > 0.f) {
          lastj = i;
          base_last = run;
          if (nr > target) { found = i; base = run; }
        }
        run = nr;
      }
      if (found < 0) { found = lastj; base = base_last; }
      int f = pl.flags | sm.flags_extra;
      if (!use_w) f |= SPEC_ST_R_ZERO;
      sm.owner = lane * per + found;
      sm.base = base;
      sm.target = target;
      sm.flags = f;
      sm.mass_out = pair ? (use_w ? R : 0.f) : Pm;
      sm.token = -1;
      sm.lastpos = -1;
    }
  }
  __syncthreads();
  const bool draw_p = (sm.flags & SPEC_ST_R_ZERO) != 0 || !pair;
  const float target = sm.target;
  const int oj = sm.owner;
  const int wlen = geo.dchunk / kWarps;
  const int64_t lo = int64_t(oj / kWarps) * geo.dchunk + int64_t(oj % kWarps) * wlen;
  const int64_t hi = lo + wlen < a.V ? lo + wlen : a.V;
  const raw* rp = sq.prow(pl.m, a.V);
  const raw* rq = pair ? sq.Q + int64_t(pl.m) * a.V : rp;
  float run = sm.base;
  for (int64_t e0 = lo; e0 < hi; e0 += kStep) {
    const int64_t e = e0 + int64_t(tid) * N;
    const uint4 vp = vec_at<E, kVec>(rp, e, hi), vq = vec_at<E, kVec>(rq, e, pair ? hi : 0);
    float s = 0.f;
    {
      float wv[N], pv[N];
      weights<E, kTrunc>(vp, vq, pair, sq.k, pl.mkp, pl.invp, pl.mkq, pl.invq, wv, pv, pl.taup, pl.tauq);
#pragma unroll
      for (int j = 0; j < N; ++j) s = __fadd_rn(s, draw_p ? pv[j] : wv[j]);
    }
    const float inc = warp_incl_scan(s);
    if (lane == 31) sm.wp[warp].x = inc;
    __syncthreads();
    float wex = run;   // running weight before this warp's first vector
    for (int i = 0; i < warp; ++i) wex = __fadd_rn(wex, sm.wp[i].x);
    float stot = run;
    for (int i = 0; i < kWarps; ++i) stot = __fadd_rn(stot, sm.wp[i].x);
    const float at = __fadd_rn(wex, inc);   // running weight through this vector
    const unsigned h = __ballot_sync(kFull, s > 0.f && at > target);
    const unsigned ps = __ballot_sync(kFull, s > 0.f);
    __syncthreads();   // every warp has read sm.wp
    if (lane == 0) sm.wp[warp] = make_float2(__int_as_float(int(h != 0)), __int_as_float(int(ps != 0)));
    __syncthreads();
    int hw = -1, pw = -1;
    for (int i = 0; i < kWarps; ++i) {
      if (hw < 0 && __float_as_int(sm.wp[i].x)) hw = i;
      if (__float_as_int(sm.wp[i].y)) pw = i;
    }
    // the thread holding the target (the first hit), or the last with weight for the fallback
    const int sel_w = hw >= 0 ? hw : pw;
    if (sel_w == warp) {
      const unsigned mask = hw >= 0 ? h : ps;
      const int sl = hw >= 0 ? __ffs(mask) - 1 : 31 - __clz(mask);
      if (lane == sl) {
        // the same weights again, from the vectors kept in registers
        float wv[N], pv[N];
        weights<E, kTrunc>(vp, vq, pair, sq.k, pl.mkp, pl.invp, pl.mkq, pl.invq, wv, pv, pl.taup, pl.tauq);
        float r = __fsub_rn(at, s);
        int t = -1, lp_ = -1;
#pragma unroll
        for (int j = 0; j < N; ++j) {
          const float wj = draw_p ? pv[j] : wv[j];
          r = __fadd_rn(r, wj);
          if (wj > 0.f) {
            lp_ = int(e) + j;
            if (t < 0 && r > target) t = int(e) + j;
          }
        }
        if (hw >= 0) sm.token = t >= 0 ? t : lp_;   // a hit vector holds the token up to rounding
        else sm.lastpos = lp_;
      }
    }
    run = stot;
    __syncthreads();
    if (sm.token >= 0) break;
  }
  const int m = pl.m;
  const int tok = sm.token >= 0 ? sm.token : (sm.lastpos >= 0 ? sm.lastpos : int(lo));
  if (tid == 0) {
    int hist;
    const int cf = commit_apply(a, b, m, cin, &hist);
    sm.hist = hist;
    if (a.diag) a.diag[int64_t(b) * (2 * gmax + 1) + 2 * gmax] = sm.mass_out;
    a.num_accepted[b] = m;
    if (a.status) a.status[b] = (sm.flags | cf) & 0xff;
    uint64_t* pw = w.planw + int64_t(b) * 4;
    for (int i = 0; i < 4; ++i) pw[i] = 0;
    w.bdone[b] = 0;
  }
  __syncthreads();
  // gmax < kThreads: thread i writes output i
  if (tid <= gmax) put_output(a, b, tid, m, tid < m ? dtok : (tid == m ? tok : -1), sm.hist);
  for (int c = tid; c < geo.DCL; c += kThreads) w.state[int64_t(b) * geo.DCL + c] = kChunkFree;
  __syncthreads();
}

// one draw chunk: the (residual, p) masses of its kWarps sub-ranges; the last draw chunk of b
// to finish selects
template <class E, bool kVec, bool kMixed, bool kTrunc = false>
__device__ void draw_chunk(const Args& a, const Geo& geo, const Work& w, const Seq<E, kMixed>& sq, const PlanRec pl,
                           int dc, Shared& sm) {
  using raw = typename E::raw;
  constexpr int N = E::kPerVec;
  constexpr int kStep = 32 * kDrawVec * N;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int b = sq.b;
  const bool pair = pl.pair != 0;
  const raw* rp = sq.prow(pl.m, a.V);
  const raw* rq = pair ? sq.Q + int64_t(pl.m) * a.V : rp;
  const int wlen = geo.dchunk / kWarps;
  const int64_t lo = int64_t(dc) * geo.dchunk + int64_t(warp) * wlen;
  const int64_t hi = lo + wlen < a.V ? lo + wlen : a.V;
  // the chunk's arrival is counted as it starts (the round trip hidden behind its loads): the
  // last to arrive selects, polling (bounded) the masses of chunks that arrived before it, which
  // are therefore being reduced
  int arrived = 0;
  if (tid == 0) arrived = atom_add_relaxed(&w.bdone[b], 1);
  float2 ws2 = make_float2(0.f, 0.f), ps2 = ws2;
  for (int64_t e0 = lo; e0 < hi; e0 += kStep) {
    uint4 vp[kDrawVec], vq[kDrawVec];
#pragma unroll
    for (int q = 0; q < kDrawVec; ++q) {
      const int64_t e = e0 + int64_t(q * 32 + lane) * N;
      vp[q] = vec_at<E, kVec>(rp, e, hi);
      vq[q] = vec_at<E, kVec>(rq, e, pair ? hi : 0);
    }
#pragma unroll
    for (int q = 0; q < kDrawVec; ++q) {
      float wv[N], pv[N];
      weights<E, kTrunc>(vp[q], vq[q], pair, sq.k, pl.mkp, pl.invp, pl.mkq, pl.invq, wv, pv, pl.taup, pl.tauq);
#pragma unroll
      for (int h = 0; h < N / 2; ++h) {
        ws2 = add2(ws2, make_float2(wv[2 * h], wv[2 * h + 1]));
        ps2 = add2(ps2, make_float2(pv[2 * h], pv[2 * h + 1]));
      }
    }
  }
  const float ws = warp_sum(__fadd_rn(ws2.x, ws2.y));
  const float ps = warp_sum(__fadd_rn(ps2.x, ps2.y));
  // each warp publishes its sub-range's word, (residual, -p): the sign bit of -p (p >= 0)
  // makes it nonzero; the selector polls the words, so no fence orders them
  if (lane == 0)
    st_relaxed_u64(&w.mass[(int64_t(b) * geo.DCL + dc) * kWarps + warp], pack_word(__float_as_uint(ws), __float_as_uint(-ps)));
  __syncthreads();
  if (tid == 0) sm.last = arrived == geo.DCL - 1;
  __syncthreads();
  if (sm.last) select<E, kVec, kMixed, kTrunc>(a, geo, w, sq, pl, sm);
}

// ------------------------------------------------------------------------------------------
// decider: combine the partials of sequence b, decide, then greedy result or the plan
// ------------------------------------------------------------------------------------------


// Entered by every thread of the block whose A unit arrived last (the arrival count reached
// its total), after a block barrier.  The partials and draft logits are taken from their
// published words.
template <class E, bool kVec, bool kMixed>
__device__ void decide(const Args& a, const Geo& geo, const Work& w, const Seq<E, kMixed>& sq, Shared& sm) {
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int b = sq.b, g = sq.g, gmax = a.gmax, CL = geo.CL;
  const float k = sq.k;
  if (tid == 0) sm.flags_extra = 0;
  __syncthreads();
  // the per-draft inputs first: they do not depend on the combine below.  Every read is
  // issued before any is waited on.
  int d = -1;
  float u = 0.f, xp = 0.f, xq = 0.f;
  uint64_t* xdp = w.xd + int64_t(b) * geo.nslots + lane;
  uint64_t* xdq = xdp + gmax + 1;
  uint64_t vxp = 0, vxq = 0;
  const bool drafts = warp == 0 && lane < g;
  if (drafts) {
    d = __ldg(&a.draft_tokens[int64_t(b) * gmax + lane]);
    if (sq.sampling) {
      u = __ldg(&a.u_accept[int64_t(b) * gmax + lane]);
      vxp = ld_relaxed_u64(xdp);
      vxq = ld_relaxed_u64(xdq);
    }
  }
  // a greedy sequence (or tree) is committed here: its lengths are loaded with the rest
  const CommitIn cin = (tid == 0 && !sq.sampling) ? commit_load(a, b) : CommitIn{0, 0, 0};
  // The row partials, a batch of rows at a time: every word of the batch is loaded at once (a
  // thread per word) and staged in shared memory, then one warp per row combines them, lanes
  // taking chunks c and c + 32 (at most 64 chunks).
  uint64_t* part = w.part + int64_t(b) * geo.nslots * CL;
  const float2 none = make_float2(-INFINITY, sq.sampling ? 0.f : __int_as_float(INT_MAX));
  auto unpack = [&](uint64_t v) {
    const uint32_t hi = uint32_t(v >> 32);
    return make_float2(__uint_as_float(uint32_t(v)), sq.sampling ? __uint_as_float(hi) : __int_as_float(int(~hi)));
  };
  const int per_batch = kPartBuf / CL;   // rows per batch (CL <= kMaxChunks < kPartBuf)
  for (int s0 = 0; s0 < geo.nslots; s0 += per_batch) {
    const int s1 = s0 + per_batch < geo.nslots ? s0 + per_batch : geo.nslots;
    const int nw = (s1 - s0) * CL;
    uint64_t* pb = part + s0 * CL;
    uint64_t v[kPartBuf / kThreads];
#pragma unroll
    for (int j = 0; j < kPartBuf / kThreads; ++j) {
      const int i = tid + j * kThreads;
      v[j] = (i < nw && sq.slot_valid(s0 + i / CL, gmax)) ? ld_relaxed_u64(&pb[i]) : 0;
    }
#pragma unroll
    for (int j = 0; j < kPartBuf / kThreads; ++j) {
      const int i = tid + j * kThreads;
      if (i < nw) sm.pbuf[i] = sq.slot_valid(s0 + i / CL, gmax) ? unpack(settle_word(&pb[i], v[j], sm)) : none;
    }
    __syncthreads();
  for (int slot = s0 + warp; slot < s1; slot += kWarps) {
    if (!sq.slot_valid(slot, gmax)) continue;
    const float2* pp = sm.pbuf + (slot - s0) * CL;
    const float2 p0 = lane < CL ? pp[lane] : none;
    const float2 p1 = lane + 32 < CL ? pp[lane + 32] : none;
    if (sq.sampling) {
      const float M = warp_max(fmaxf(p0.x, p1.x));
      // a chunk without a finite logit adds its sum as it is (0, or NaN: see warp_stats)
      const float t0 = p0.x == -INFINITY ? p0.y : __fmul_rn(p0.y, ex2(__fmul_rn(p0.x - M, k)));
      const float t1 = p1.x == -INFINITY ? p1.y : __fmul_rn(p1.y, ex2(__fmul_rn(p1.x - M, k)));
      const float S = warp_sum(__fadd_rn(t0, t1));
      if (lane == 0) {
        sm.rowM[slot] = M;
        sm.rowInvS[slot] = __frcp_rn(S);
        // no finite max, or a NaN in the row: it defines no distribution
        if (!(isfinite(M) && isfinite(S))) atomicOr(&sm.flags_extra, SPEC_ST_BAD_ROW);
      }
    } else {
      float bv = p0.x;
      int bi = __float_as_int(p0.y);
      if (better(p1.x, __float_as_int(p1.y), bv, bi)) { bv = p1.x; bi = __float_as_int(p1.y); }
      warp_argmax(bv, bi);
      if (lane == 0) sm.rowArg[slot] = bi;
    }
  }
    __syncthreads();   // the buffer is refilled by the next batch
  }
  if (drafts && sq.sampling) {
    // published for every draft row: the logit at d, or a marker when d is outside the row
    xp = __uint_as_float(uint32_t(settle_word(xdp, vxp, sm)));
    xq = __uint_as_float(uint32_t(settle_word(xdq, vxq, sm)));
  }
  if (tid < 2) sm.taken[tid] = 0u;
  __syncthreads();
  if (!kMixed && a.parents) {
    // Greedy tree verification (tutorial §5.3): node j (1..g) carries draft_tokens[b][j-1]
    // and hangs below parents[b][j-1] (0 is the root); it is accepted iff its parent is and
    // its token is the argmax of the parent's row.  The path ends at the deepest accepted
    // node, the lowest index among equal depths.  Parents precede their children, so one
    // pass in index order settles every node.
    for (int j = tid; j < g; j += kThreads) {
      sm.tpar[j + 1] = a.parents[int64_t(b) * gmax + j];
      sm.ttok[j + 1] = a.draft_tokens[int64_t(b) * gmax + j];
    }
    __syncthreads();
    if (tid == 0) {
      int f = sq.flags | sm.flags_extra;
      sm.tacc[0] = 1;
      sm.tdep[0] = 0;
      int best = 0, bestd = 0;
      for (int j = 1; j <= g; ++j) {
        const int par = sm.tpar[j], d = sm.ttok[j];
        sm.tacc[j] = 0;
        sm.tdep[j] = 0;
        if (par < 0 || par >= j) {
          f |= SPEC_ST_BAD_TREE;
          continue;
        }
        const int dep = sm.tdep[par] + 1;
        sm.tdep[j] = (unsigned char)dep;
        if (!sm.tacc[par]) continue;
        if (d < 0 || int64_t(d) >= a.V) {
          f |= SPEC_ST_BAD_DRAFT;
          continue;
        }
        if (d == sm.rowArg[par]) {
          sm.tacc[j] = 1;
          if (dep > bestd) {
            best = j;
            bestd = dep;
          }
        }
      }
      int j = best;
      for (int i = bestd - 1; i >= 0; --i) {
        sm.tpath[i] = j;
        j = sm.tpar[j];
      }
      sm.m = bestd;
      sm.flags = f;
      sm.tbest = best;
    }
    __syncthreads();
    const int m = sm.m;
    if (tid == 0) {
      // the round's commit when the call carries one: the lengths advance by the path's m
      // (+1), the path's tokens are appended (the caller compacts its cache by path_nodes)
      int hist;
      const int cf = commit_apply(a, b, m, cin, &hist);
      sm.hist = hist;
      a.num_accepted[b] = m;
      if (a.status) a.status[b] = sm.flags | cf;
      w.cnt[b] = 0;
    }
    __syncthreads();
    for (int i = tid; i <= gmax; i += kThreads) {
      int v = -1;
      if (i < m) v = sm.ttok[sm.tpath[i]];
      else if (i == m) v = sm.rowArg[sm.tbest];
      put_output(a, b, i, m, v, sm.hist);
    }
    if (a.path_nodes)
      for (int i = tid; i < gmax; i += kThreads) a.path_nodes[int64_t(b) * gmax + i] = i < m ? sm.tpath[i] : -1;
    __syncthreads();
    return;
  }
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
      int f = sq.flags | sm.flags_extra;
      if (m < g && ((bad >> m) & 1u)) f |= SPEC_ST_BAD_DRAFT;
      sm.m = m;
      sm.flags = f;
    }
  }
  __syncthreads();
  const int m = sm.m;
  if (!sq.sampling) {
    if (tid == 0) {
      int hist;
      const int cf = commit_apply(a, b, m, cin, &hist);
      sm.hist = hist;
      a.num_accepted[b] = m;
      if (a.status) a.status[b] = sm.flags | cf;
      w.cnt[b] = 0;
    }
    __syncthreads();
    // thread i < m is lane i of warp 0, which holds d_i
    if (tid <= gmax) put_output(a, b, tid, m, tid < m ? d : (tid == m ? sm.rowArg[m] : -1), sm.hist);
    if (a.diag)
      for (int i = tid; i < 2 * gmax + 1; i += kThreads) a.diag[int64_t(b) * (2 * gmax + 1) + i] = NAN;
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
    sm.plan = pr;
    w.cnt[b] = 0;
    // four published words, no fence: a draw unit polls each (plan_words)
    uint64_t* pw = w.planw + int64_t(b) * 4;
    st_relaxed_u64(pw + 1, pack_word(__float_as_uint(pr.invp), 1u));
    st_relaxed_u64(pw + 2, pack_word(__float_as_uint(pr.mkq), 1u));
    st_relaxed_u64(pw + 3, pack_word(__float_as_uint(pr.invq), 1u));
    st_relaxed_u64(pw, pack_word(uint32_t(ready_word(pr)), __float_as_uint(pr.mkp)));
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
    // A row past num_draft (or a draft row of a greedy sequence) is never read: in ragged or
    // mixed batches such rows can be a large share of the grid.
    const raw* row = slot <= a.gmax
                         ? target_row<E>(a, b, slot)
                         : static_cast<const raw*>(a.draft) + (int64_t(b) * a.gmax + (slot - a.gmax - 1)) * a.V;
    const int64_t lo = int64_t(c) * geo.chunk;
    const int64_t hi = lo + geo.chunk < a.V ? lo + geo.chunk : a.V;
    auto fetch = [&](Tile<E, kVec>& t, int64_t e0) {
      if (e0 + kPass <= hi) t.load_full(row, e0, tid);
      else t.load(row, e0, hi, tid);
    };
    Tile<E, kVec> t0, t1;
    const Seq<E, kMixed> sq(a, b);
    if (!sq.slot_valid(slot, a.gmax)) return;
    if (lo < hi) fetch(t0, lo);
    if (lo + kPass < hi) fetch(t1, lo + kPass);
    // The arrival is counted now, its round trip hidden behind the row: the unit that arrives
    // last decides once its own row is done, and waits (bounded, in settle_word) for the
    // partials of units that arrived before it and are still reading.  Those have arrived, so
    // they are running: the wait never depends on a block that has not started.
    int arrived = 0;
    if (tid == 0) arrived = atom_add_relaxed(&w.cnt[b], 1);
    // the logit at this row's draft id, if it lies in this chunk: fetched once, up front
    const int i = slot <= a.gmax ? slot : slot - a.gmax - 1;
    bool has_d = false, no_d = false;
    float xv = 0.f;
    if (tid == 0 && sq.sampling && i < sq.g) {
      const int d = __ldg(&a.draft_tokens[int64_t(b) * a.gmax + i]);
      has_d = int64_t(d) >= lo && int64_t(d) < hi;
      no_d = c == 0 && (d < 0 || int64_t(d) >= a.V);   // no chunk holds it: chunk 0 says so
      if (has_d) xv = E::at(row, d);
    }
    float rm = -INFINITY, rs = 0.f;
    int ri = INT_MAX;
    constexpr bool kKeep = kVec && !kMixed;   // the greedy-only kernel has the registers to spare
    KeptTile<E> kept;
    auto consume = [&](const Tile<E, kVec>& t, int64_t e0) {
      if constexpr (kKeep) {
        kept.offer(t, e0);
      } else {
        if (sq.sampling) thread_stats(t, sq.k, rm, rs);
        else tile_argmax(t, e0, tid, rm, ri);
      }
    };
    {
      // two tiles in registers, both passes already in flight: each is refilled with the
      // pass after next as soon as it has been reduced
      for (int64_t e0 = lo; e0 < hi; e0 += 2 * kPass) {
        consume(t0, e0);
        if (e0 + 2 * kPass < hi) fetch(t0, e0 + 2 * kPass);
        if (e0 + kPass >= hi) break;
        consume(t1, e0 + kPass);
        if (e0 + 3 * kPass < hi) fetch(t1, e0 + 3 * kPass);
      }
    }
    if constexpr (kKeep) kept.settle(tid, rm, ri);
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
        // published without a fence (see st_relaxed_u64); the arrival count only elected the
        // decider, which polls the words themselves
        if (has_d || no_d)
          st_relaxed_u64(&w.xd[int64_t(b) * geo.nslots + slot], pack_word(canon_bits(has_d ? xv : NAN), has_d ? 1u : 2u));
        st_relaxed_u64(&w.part[(int64_t(b) * geo.nslots + slot) * geo.CL + c],
                       sq.sampling ? pack_word(canon_bits(p.x), __float_as_uint(p.y))
                                   : pack_word(canon_bits(p.x), ~uint32_t(__float_as_int(p.y))));
        sm.last = arrived == geo.CL * sq.nrows() - 1;
      }
    }
    __syncthreads();
    if (sm.last) decide<E, kVec, kMixed>(a, geo, w, sq, sm);
    return;
  }

  if constexpr (kMixed) {
    // ---------------- B unit: draw chunk dc of the sequence of this group --------------------
    const int dc = (y - geo.nslots) * geo.CL + x;
    const int bl = draw_group_seq(int(blockIdx.z), geo.b1 - geo.b0, geo.delta, geo.ndefer);
    if (dc >= geo.DCL || bl < 0) return;
    const int b = geo.b0 + bl;
    const Seq<E, kMixed> sq(a, b);
    // the plan's first word is read while the sequence's metadata loads are still in flight
    uint64_t* pw = w.planw + int64_t(b) * 4;
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    if (tid == 0) {
      w0 = ld_relaxed_u64(pw);
      w1 = ld_relaxed_u64(pw + 1);
      w2 = ld_relaxed_u64(pw + 2);
      w3 = ld_relaxed_u64(pw + 3);
    }
    if (!sq.sampling) return;
    if (tid == 0) {
      int* st = &w.state[int64_t(b) * geo.DCL + dc];
      // optional, bounded wait for the plan; correctness does not depend on it
      int it = 0, ns = 64;
      while (uint32_t(w0) == 0 && it < kPlanWaitIters) {
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;
        ++it;
        w0 = ld_relaxed_u64(pw);
      }
      bool mine = false;
      if (uint32_t(w0) != 0) {
        // the plan is out: the decider takes only given-up chunks, so this one stays ours
        // without a claim
        mine = true;
      } else if (atom_cas(st, kChunkFree, kChunkGivenUp) == kChunkFree) {
        // given up; if the plan appeared meanwhile, take the chunk back unless the decider has
        __threadfence();
        w0 = ld_relaxed_u64(pw);
        if (uint32_t(w0) != 0) mine = atom_cas(st, kChunkGivenUp, kChunkMine) == kChunkGivenUp;
      }
      if (mine) {
        // the other three words were stored before the first, in no guaranteed order: each
        // is taken once it is there (bounded)
        const long long t0 = global_ns();
        while ((w1 == 0 || w2 == 0 || w3 == 0) && global_ns() - t0 < kWaitNs) {
          if (w1 == 0) w1 = ld_relaxed_u64(pw + 1);
          if (w2 == 0) w2 = ld_relaxed_u64(pw + 2);
          if (w3 == 0) w3 = ld_relaxed_u64(pw + 3);
        }
        const int rdy = int(uint32_t(w0));
        sm.plan.m = rdy & 0xffff;
        sm.plan.pair = (rdy >> 16) & 1;
        sm.plan.flags = (rdy >> 20) & 0xff;
        sm.plan.g = sq.g;
        sm.plan.mkp = __uint_as_float(uint32_t(w0 >> 32));
        sm.plan.invp = __uint_as_float(uint32_t(w1));
        sm.plan.mkq = __uint_as_float(uint32_t(w2));
        sm.plan.invq = __uint_as_float(uint32_t(w3));
        // never fails for a well-formed workspace; keeps every read in bounds
        if (w1 == 0 || w2 == 0 || w3 == 0 || sm.plan.m > sq.g || (sm.plan.pair && sm.plan.m >= sq.g)) {
          mine = false;
          if (a.status) atomicOr(&a.status[b], SPEC_ST_TIMEOUT);
        }
      }
      sm.go = mine;
    }
    __syncthreads();
    if (!sm.go) return;
    const PlanRec pl = sm.plan;
    draw_chunk<E, kVec, kMixed>(a, geo, w, sq, pl, dc, sm);
  }
}

// ------------------------------------------------------------------------------------------
// truncated sampling: per-row thresholds, then the decisions, then the draw
// ------------------------------------------------------------------------------------------
//
// The same truncation on both sides (the "M013" card §10 and the nxmr note: temperature,
// top-p or any other logits processing must show in p and q).  For every valid row of a
// sampling sequence one block finds the row's max M, then the smallest kept logit tau: top-k
// keeps the logits >= the k-th largest (ties kept), top-p then keeps those >= the largest t
// whose kept mass at or above t reaches top_p times the top-k-kept mass.  Both thresholds are
// found exactly by counting the ids of each order-preserving 16-bit key of the bf16 logits in
// windows of 256 keys from the top: all ids of one key share one logit, so a key's mass is
// its count times that logit's mass, in fixed point (2^-40 units, summed in integers, so every
// run gives the same bits).  A sample of the row places the first window before the one pass
// that also takes M; further windows, if any, are further passes.  The row's normaliser is the
// kept mass; p'(v) = 0 below tau.

struct TruncArgs {
  const int32_t* top_k;   // [B] or null
  const float* top_p;     // [B] or null
};

struct __align__(16) RowInfo {
  float mk;     // M * k
  float invs;   // 1 / kept mass
  float tau;    // smallest kept logit (-inf: everything kept)
  int arg;      // greedy rows: lowest-id argmax
};

constexpr float kMassUnit = 1099511627776.0f;   // 2^40
constexpr uint32_t kGuardKeys = 96;        // fused window's top above the estimated max
constexpr uint32_t kFusedWidth = 256; // keys the fused pass counts: one window
constexpr int kSampleRuns = 4;     // runs of kThreads vectors the estimate reads
constexpr int kTruncDrawChunk = 32768;  // ids per draw unit of the truncated draw

// order-preserving 16-bit key of a bf16 logit; -0 is taken as +0 so equal values share a key
__device__ __forceinline__ uint32_t key16(uint32_t bits) {
  bits &= 0xffffu;
  if (bits == 0x8000u) bits = 0;
  return (bits & 0x8000u) ? (~bits & 0xffffu) : (bits | 0x8000u);
}
__device__ __forceinline__ float key16_value(uint32_t key) {
  const uint32_t bits = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
  return __uint_as_float(bits << 16);
}

constexpr int kQueueSlots = 64;      // per warp: vectors queued for counting by the fused pass

struct TruncShared {
  unsigned cnt[2][256];          // window counts: [0] a pass's window (the fused pass's too); [1] is
                                 // cleared with it and stays empty at a fused width of 256 keys
  uint4 cq[kWarps][kQueueSlots]; // the fused pass's per-warp queues of vectors that reach the window
  float wm[kWarps];
  int wi[kWarps];
  unsigned long long wtot[kWarps];
  int res_d;
  uint32_t res_cnt;
  unsigned long long res_mass;
};

// The key of -inf; smaller keys are NaN patterns, which no window counts.
constexpr uint32_t kKeyNegInf = 0x7fu;

// fixed-point sum over the block of one value per thread (a fixed order, so fixed bits)
__device__ unsigned long long block_sum_u64(unsigned long long s, TruncShared& ts) {
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(kFull, s, o);
  const int lane = int(threadIdx.x) & 31, warp = int(threadIdx.x) >> 5;
  if (lane == 0) ts.wtot[warp] = s;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < kWarps; ++i) t += ts.wtot[i];
  __syncthreads();
  return t;
}

// the block's max of one value per thread, returned to every thread
__device__ float block_max_f32(float m, TruncShared& ts) {
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) ts.wm[threadIdx.x >> 5] = m;
  __syncthreads();
  float r = ts.wm[0];
  for (int i = 1; i < kWarps; ++i) r = fmaxf(r, ts.wm[i]);
  __syncthreads();
  return r;
}

// Visits every id of a row once: fn(x, bits, id) per element, eight 16-byte vectors per thread
// per step, coalesced across the block.
template <bool kVec, class Fn>
__device__ __forceinline__ void for_each_bf16(const uint16_t* row, int64_t V, Fn fn) {
  constexpr int kVecs = 8;
  constexpr int kStep = kThreads * 8 * kVecs;
  for (int64_t e0 = 0; e0 < V; e0 += kStep) {
    uint4 v[kVecs];
#pragma unroll
    for (int q = 0; q < kVecs; ++q) v[q] = vec_at<Bf16, kVec>(row, e0 + int64_t(q * kThreads + int(threadIdx.x)) * 8, V);
#pragma unroll
    for (int q = 0; q < kVecs; ++q) {
      const int64_t e = e0 + int64_t(q * kThreads + int(threadIdx.x)) * 8;
      const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
      if (e + 8 <= V) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t bits = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
          fn(__uint_as_float(bits << 16), bits, int(e + j));
        }
      } else {
        for (int j = 0; j < 8 && e + j < V; ++j) {
          const uint32_t bits = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
          fn(__uint_as_float(bits << 16), bits, int(e + j));
        }
      }
    }
  }
}

// Visits every 16-byte vector of a row once: fn(v, nvalid), nvalid = the ids of v inside the
// row (8 but at a ragged tail), eight vectors per thread per step, coalesced across the block.
// Vectors wholly past the row are skipped, unless kAll: then every thread calls fn the same
// number of times (a warp can vote in fn), past the row with vectors of -inf and nvalid 0.
// With kAll (the fused pass, whose fn is light) the whole steps go by halves of four vectors
// per thread, the next half's loads issued before this half is visited.
template <bool kVec, class Fn, bool kAll = false>
__device__ __forceinline__ void for_each_vec(const uint16_t* row, int64_t V, Fn fn) {
  constexpr int kVecs = 8;
  constexpr int kStep = kThreads * 8 * kVecs;
  const int tid = int(threadIdx.x);
  int64_t e0 = 0;
  if constexpr (kVec && kAll) {
    // whole half steps, the next one's loads in flight while this one is visited
    constexpr int kH = kVecs / 2;
    constexpr int kHStep = kThreads * 8 * kH;
    if (kHStep <= V) {
      uint4 cur[kH];
#pragma unroll
      for (int q = 0; q < kH; ++q) cur[q] = ld_stream(row + int64_t(q * kThreads + tid) * 8);
      for (;;) {
        const int64_t en = e0 + kHStep;
        const bool more = en + kHStep <= V;
        uint4 nxt[kH];
        if (more) {
#pragma unroll
          for (int q = 0; q < kH; ++q) nxt[q] = ld_stream(row + en + int64_t(q * kThreads + tid) * 8);
        }
#pragma unroll
        for (int q = 0; q < kH; ++q) fn(cur[q], 8);
        e0 = en;
        if (!more) break;
#pragma unroll
        for (int q = 0; q < kH; ++q) cur[q] = nxt[q];
      }
    }
  } else if constexpr (kVec) {
    // whole steps: every vector inside the row (V is a multiple of 8 here), no checks
    for (; e0 + kStep <= V; e0 += kStep) {
      uint4 v[kVecs];
#pragma unroll
      for (int q = 0; q < kVecs; ++q) v[q] = ld_stream(row + e0 + int64_t(q * kThreads + tid) * 8);
#pragma unroll
      for (int q = 0; q < kVecs; ++q) fn(v[q], 8);
    }
  }
  for (; e0 < V; e0 += kStep) {
    uint4 v[kVecs];
#pragma unroll
    for (int q = 0; q < kVecs; ++q) v[q] = vec_at<Bf16, kVec>(row, e0 + int64_t(q * kThreads + tid) * 8, V);
#pragma unroll
    for (int q = 0; q < kVecs; ++q) {
      const int64_t e = e0 + int64_t(q * kThreads + tid) * 8;
      if (kAll || e < V) fn(v[q], e >= V ? 0 : (V - e < 8 ? int(V - e) : 8));
    }
  }
}

// The window of one pass: keys hi-width+1..hi, bin d = hi - key.
struct Window {
  uint32_t hi;
  uint32_t width;
  uint32_t blo;    // fast form: the bf16 code of the lowest key
  bool fast;       // the window lies above +0: bf16 codes order like the values there
  float vlo, vhi;  // the window's lowest and highest values
  __device__ Window(uint32_t h, uint32_t w) : hi(h), width(w) {
    fast = h > 0x8000u + w - 1u;
    blo = fast ? h - (w - 1u) - 0x8000u : 0u;
    vhi = key16_value(h);
    vlo = h >= w - 1u + kKeyNegInf ? key16_value(h - (w - 1u)) : -INFINITY;
  }
};

// adds 1 to the shared word at addr when t < width, without a branch
__device__ __forceinline__ void count_if(uint32_t t, uint32_t width, uint32_t addr) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.lt.u32 p, %0, %1;\n\t@p red.shared.add.u32 [%2], 1;\n\t}" ::"r"(t), "r"(width),
               "r"(addr));
}

// One vector's part of a window pass.  kFast: a logit is in the window iff its code minus blo
// is below the width (unsigned; negative logits wrap far above), its bin is width-1 minus
// that, and padding (-inf) is never in it; otherwise the order-preserving key decides, ids past
// nvalid skipped.  With kBelow, the ids under the window add their mass to f, in id order.
// With kNext, xb keeps the largest logit under the window (where the next window can start).
template <bool kFast, bool kBelow, bool kNext = false>
__device__ __forceinline__ void window_vec(const uint4& v, int nvalid, const Window& win, float k, float mk,
                                           unsigned* cnt, float& f, float& xb) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint32_t clast = smem_addr(cnt) + 4u * (win.width - 1u);   // bin width-1: code blo
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t bits = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
    if constexpr (kFast) {
      const uint32_t t = bits - win.blo;
      count_if(t, win.width, clast - 4u * t);
      if constexpr (kBelow || kNext) {
        const float x = __uint_as_float(bits << 16);
        if constexpr (kBelow) f = __fadd_rn(f, x < win.vlo ? ex2(fmaf(x, k, -mk)) : 0.f);
        if constexpr (kNext) xb = fmaxf(xb, x < win.vlo ? x : -INFINITY);
      }
    } else {
      if (j >= nvalid) break;
      const float x = __uint_as_float(bits << 16);
      if (x < win.vlo) {
        if constexpr (kBelow) f = __fadd_rn(f, ex2(fmaf(x, k, -mk)));
        if constexpr (kNext) xb = fmaxf(xb, x);
      } else if (x <= win.vhi) {
        atomicAdd(&cnt[win.hi - key16(bits)], 1u);
      }
    }
  }
}

// One window pass: bin d counts the ids of key hi - d (d < 256).  Every id of one key has the
// same logit, so a bin's mass is its count times that logit's exp: counting is all the pass does
// per id inside the window (one 32-bit shared reduction), ids above it are skipped, and with `below`
// the ids under it add their mass to a per-thread float sum, returned as the block's fixed-point
// total.
// `next` receives the key of the largest logit under the window (the key of -inf when there is
// none): no key between it and the window holds an id, so the next window can start there.
template <bool kVec>
__device__ unsigned long long trunc_window(const uint16_t* row, int64_t V, uint32_t hi, bool below, float k,
                                           float mk, TruncShared& ts, uint32_t& next) {
  unsigned* cnt = ts.cnt[0];
  for (int i = int(threadIdx.x); i < 256; i += kThreads) cnt[i] = 0;
  __syncthreads();
  const Window win(hi, 256u);
  float f = 0.f, xb = -INFINITY;
  if (win.fast) {
    if (below) for_each_vec<kVec>(row, V, [&](const uint4& v, int nv) { window_vec<true, true, true>(v, nv, win, k, mk, cnt, f, xb); });
    else for_each_vec<kVec>(row, V, [&](const uint4& v, int nv) { window_vec<true, false, true>(v, nv, win, k, mk, cnt, f, xb); });
  } else {
    if (below) for_each_vec<kVec>(row, V, [&](const uint4& v, int nv) { window_vec<false, true, true>(v, nv, win, k, mk, cnt, f, xb); });
    else for_each_vec<kVec>(row, V, [&](const uint4& v, int nv) { window_vec<false, false, true>(v, nv, win, k, mk, cnt, f, xb); });
  }
  __syncthreads();
  next = key16(__float_as_uint(block_max_f32(xb, ts)) >> 16);
  return below ? block_sum_u64(__float2ull_rn(f * kMassUnit), ts) : 0ull;
}

// Warp 0 walks the window's bins d = 0..dmax from the top: the first bin at which the running
// count (by_count) or the running fixed-point mass reaches `target`.  Each lane takes eight
// bins, the lanes' sums are scanned, and the lane holding the crossing walks its own bins.
// Leaves in ts: res_d (-1: not reached), and the count and mass of bins 0..res_d (of the whole
// window when not reached).  count(d) gives bin d's count.
template <class Count>
__device__ void trunc_scan(TruncShared& ts, Count count, uint32_t hi, int dmax, float k, float mk, bool by_count,
                           unsigned long long target) {
  if (threadIdx.x < 32) {
    const int lane = int(threadIdx.x);
    uint32_t c[8];
    unsigned long long w[8];
    uint32_t lc = 0;
    unsigned long long lw = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d = lane * 8 + j;
      c[j] = d <= dmax ? count(d) : 0u;
      w[j] = c[j] ? c[j] * (unsigned long long)__float2ull_rn(ex2(fmaf(key16_value(hi - uint32_t(d)), k, -mk)) *
                                                                kMassUnit)
                  : 0ull;
      lc += c[j];
      lw += w[j];
    }
    uint32_t ic = lc;
    unsigned long long iw = lw;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t uc = __shfl_up_sync(kFull, ic, o);
      const unsigned long long uw = __shfl_up_sync(kFull, iw, o);
      if (lane >= o) { ic += uc; iw += uw; }
    }
    const unsigned hit = __ballot_sync(kFull, by_count ? uint64_t(ic) >= target : iw >= target);
    if (hit == 0) {
      if (lane == 31) { ts.res_d = -1; ts.res_cnt = ic; ts.res_mass = iw; }
    } else if (lane == __ffs(hit) - 1) {
      uint32_t rc = ic - lc;
      unsigned long long rw = iw - lw;
      int d = lane * 8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rc += c[j];
        rw += w[j];
        if (by_count ? uint64_t(rc) >= target : rw >= target) { d = lane * 8 + j; break; }
      }
      ts.res_d = d;
      ts.res_cnt = rc;
      ts.res_mass = rw;
    }
  }
  __syncthreads();
}

// the mass (fixed point) of the whole row, all threads taking part
template <bool kVec>
__device__ unsigned long long trunc_total(const uint16_t* row, int64_t V, float k, float mk, TruncShared& ts) {
  // per thread in float, in a fixed order (so in fixed bits); in fixed point across threads
  float f = 0.f;
  // a NaN logit adds nothing (fmaxf turns its NaN argument into -inf), as in the window passes
  for_each_bf16<kVec>(row, V, [&](float x, uint32_t, int) { f = __fadd_rn(f, ex2(fmaxf(fmaf(x, k, -mk), -INFINITY))); });
  return block_sum_u64(__float2ull_rn(f * kMassUnit), ts);
}

// the fixed-point mass of 256 counted bins (bin d: key hi - d), thread d taking bin d
__device__ unsigned long long bins_mass(const unsigned* cnt, uint32_t hi, float k, float mk, TruncShared& ts) {
  static_assert(kThreads == 256, "one bin per thread");
  const int d = int(threadIdx.x);
  const unsigned c = cnt[d];
  const unsigned long long w =
      c ? c * (unsigned long long)__float2ull_rn(ex2(fmaf(key16_value(hi - uint32_t(d)), k, -mk)) * kMassUnit) : 0ull;
  return block_sum_u64(w, ts);
}

// The one pass of the fused search: the row's max (packed bf16 maxima) and the counts of a window
// fixed before the pass; with kBelow, the mass of the ids under the window relative to the
// window's lowest value (vk = that value times k; every term is at most 1), so that no max is
// needed during the pass.
// A window above +0 holds only values at or above its lowest value vlo, so a vector whose max
// is under vlo holds none of its ids.  Most vectors are such, and in the fast form the pass
// counts only the others: each warp queues them in shared memory (`q`, kQueueSlots vectors) and
// counts their ids 32 vectors at a time, one vector per lane.  The counts are integers, so the
// order in which ids are counted changes no bit.
template <bool kVec, bool kFast, bool kBelow>
__device__ __forceinline__ void fused_pass(const uint16_t* row, int64_t V, const Window& win, float k, float vk,
                                           unsigned* cnt, uint4* q, __nv_bfloat162& h, float& f) {
  if constexpr (!kFast) {
    for_each_vec<kVec>(row, V, [&](const uint4& v, int nv) {
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
      h = __hmax2(h, __hmax2(__hmax2(p2[0], p2[1]), __hmax2(p2[2], p2[3])));
      float unused = 0.f;
      window_vec<false, kBelow>(v, nv, win, k, vk, cnt, f, unused);
    });
  } else {
    static_assert(kQueueSlots == 64, "a queue holds fewer than 32 vectors between steps, 32 more per step");
    const int lane = int(threadIdx.x) & 31;
    const unsigned below_lane = (1u << lane) - 1u;
    const uint32_t clast = smem_addr(cnt) + 4u * (win.width - 1u);   // bin width-1: code blo
    const auto count8 = [&](const uint4& v) {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t t = ((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu)) - win.blo;
        count_if(t, win.width, clast - 4u * t);
      }
    };
    unsigned head = 0, tail = 0;   // the queue's counted and written ends (the same in every lane)
    const auto visit = [&](const uint4& v, int) {
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
      const __nv_bfloat162 vm = __hmax2(__hmax2(p2[0], p2[1]), __hmax2(p2[2], p2[3]));
      h = __hmax2(h, vm);
      if constexpr (kBelow) {
        // the mass under the window, id by id in id order, as window_vec takes it
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float x = __uint_as_float(((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu)) << 16);
          f = __fadd_rn(f, x < win.vlo ? ex2(fmaf(x, k, -vk)) : 0.f);
        }
      }
      // a NaN half loses to the other in __hmax2; a vector of NaN alone is never counted
      const bool hit = fmaxf(__low2float(vm), __high2float(vm)) >= win.vlo;
      const unsigned bal = __ballot_sync(kFull, hit);
      if (hit) q[(tail + unsigned(__popc(bal & below_lane))) % kQueueSlots] = v;
      tail += unsigned(__popc(bal));
      if (tail - head >= 32u) {
        __syncwarp();
        count8(q[(head + unsigned(lane)) % kQueueSlots]);
        head += 32u;
        __syncwarp();
      }
    };
    // every lane visits the same number of vectors (the ragged step's past-the-row ones too)
    for_each_vec<kVec, decltype(visit), true>(row, V, visit);
    __syncwarp();
    if (unsigned(lane) < tail - head) count8(q[(head + unsigned(lane)) % kQueueSlots]);
  }
}

// The thresholds of one row, over windows of 256 keys from key `top` (the row's max, or a key
// above it: the bins above the max are empty) down.
// top-k: the first key whose count from the top reaches k; top-p: then the first key whose
// kept mass from the top reaches top_p times the top-k-kept mass.  Both are exact: a window is
// searched key by key.  The window at the max usually holds both crossings, and its counts
// serve both searches.  window(hi, below) runs one window pass (returning the mass under the
// window when `below`); count(d) reads bin d of the last one; step(hi) gives the top of the next
// window below it (hi - 256, or the first key under the window that holds an id, skipping empty
// keys).  Every thread calls this with the same arguments and takes the same branches.  Leaves
// kmin (smallest kept key, 0: all) and kept (their fixed-point mass).
template <class WindowFn, class Count, class StepFn>
__device__ void trunc_search(TruncShared& ts, WindowFn window, Count count, StepFn step, uint32_t top, int topk,
                             float topp, bool dok, bool dop, float k, float mk, uint32_t& kmin,
                             unsigned long long& kept) {
  kmin = 0;
  kept = 0;
  uint32_t hi = top;                       // the window `count` reads
  if (dok) {
    unsigned long long above = 0;          // mass of the windows above hi
    uint32_t need = uint32_t(topk);        // ids still to count
    for (;;) {
      window(hi, false);
      trunc_scan(ts, count, hi, 255, k, mk, true, need);
      const int d = ts.res_d;
      const uint32_t c = ts.res_cnt;
      const unsigned long long w = ts.res_mass;
      __syncthreads();
      if (d >= 0) { kmin = hi - uint32_t(d); kept = above + w; break; }
      above += w;
      need -= c;
      if (hi < 256u + kKeyNegInf) { kept = above; break; }   // only with NaN logits: fewer than k ids counted
      hi = step(hi);
    }
  } else {
    // the whole row's mass: the window at the max by counts, the rest by per-thread sums
    const unsigned long long below = window(hi, true);
    trunc_scan(ts, count, hi, 255, k, mk, true, ~0ull);
    kept = ts.res_mass + below;
    __syncthreads();
  }
  if (!dop) return;
  const unsigned long long target = (unsigned long long)ceil(double(topp) * double(kept));
  unsigned long long acc = 0;
  uint32_t h = top;
  for (;;) {
    if (h != hi) { window(h, false); hi = h; }
    const int dmax = kmin == 0 ? 255 : int(min(255u, h - kmin));
    trunc_scan(ts, count, h, dmax, k, mk, false, target - acc);
    const int d = ts.res_d;
    const unsigned long long w = ts.res_mass;
    __syncthreads();
    if (d >= 0) { kmin = h - uint32_t(d); kept = acc + w; return; }
    acc += w;
    // cannot happen: the kept mass reaches the target
    if (h < 256u + kKeyNegInf || h - 256u < kmin) return;
    h = step(h);
    if (h < kmin) return;
  }
}

// Per row: greedy rows get their argmax; sampling rows their max, threshold and kept mass.
template <bool kVec>
__global__ void __launch_bounds__(kThreads, kVec ? kMinBlocks : 1) trunc_rows_kernel(const Args a, const TruncArgs t, RowInfo* info,
                                                              int nslots) {
  __shared__ TruncShared ts;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int64_t idx = int64_t(blockIdx.x);
  const int slot = int(idx % nslots), b = int(idx / nslots);
  const Seq<Bf16, true> sq(a, b);
  if (!sq.slot_valid(slot, a.gmax)) return;
  const uint16_t* row = slot <= a.gmax ? target_row<Bf16>(a, b, slot)
                                       : static_cast<const uint16_t*>(a.draft) + (int64_t(b) * a.gmax + (slot - a.gmax - 1)) * a.V;
  RowInfo* out = info + int64_t(b) * nslots + slot;
  const int64_t V = a.V;
  if (!sq.sampling) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for_each_bf16<kVec>(row, V, [&](float x, uint32_t, int id) {
      if (better(x, id, bv, bi)) { bv = x; bi = id; }
    });
    warp_argmax(bv, bi);
    if (lane == 0) { ts.wm[warp] = bv; ts.wi[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
      for (int i = 1; i < kWarps; ++i)
        if (better(ts.wm[i], ts.wi[i], bv, bi)) { bv = ts.wm[i]; bi = ts.wi[i]; }
      out->arg = bi;
    }
    return;
  }
  const float k = sq.k;
  const int topk = t.top_k ? t.top_k[b] : 0;
  const float topp = t.top_p ? t.top_p[b] : 1.f;
  const bool dok = topk > 0 && int64_t(topk) < V;
  const bool dop = topp > 0.f && topp < 1.f;
  // An estimate of the row's max from kSampleRuns runs of kThreads vectors spread over the row fixes
  // the window of the one pass: kFusedWidth keys from kGuardKeys keys above the estimate.
  float ms;
  {
    const int64_t nvec = (V + 7) / 8;
    const int64_t stride = nvec / kSampleRuns > kThreads ? nvec / kSampleRuns : int64_t(kThreads);
    __nv_bfloat162 h = __floats2bfloat162_rn(-INFINITY, -INFINITY);
#pragma unroll
    for (int q = 0; q < kSampleRuns; ++q) {
      const int64_t vi = int64_t(q) * stride + tid;
      if (vi < nvec) {
        const uint4 v = vec_at<Bf16, kVec>(row, vi * 8, V);
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
        h = __hmax2(h, __hmax2(__hmax2(p2[0], p2[1]), __hmax2(p2[2], p2[3])));
      }
    }
    ms = block_max_f32(fmaxf(__low2float(h), __high2float(h)), ts);
  }
  const uint32_t top = key16(__float_as_uint(ms) >> 16) + kGuardKeys;
  const bool fused = top <= 0xff7fu;       // the window stays among finite values
  float M = -INFINITY;
  uint32_t kmin = 0;                       // smallest kept key (0: everything)
  unsigned long long kept = 0;             // mass of the keys >= kmin
  bool done = false;
  bool bad = false;                        // no finite max: the row defines no distribution
  if (fused) {
    const Window win(top, kFusedWidth);
    const bool below = !dok;               // the whole row's mass is wanted
    const float vk = __fmul_rn(win.vlo, k);
    unsigned* cnt = &ts.cnt[0][0];         // [0]: keys top..top-255 ([1] stays empty at this width)
    for (int i = tid; i < 512; i += kThreads) cnt[i] = 0;
    __syncthreads();
    __nv_bfloat162 h = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    float f = 0.f;
    uint4* q = ts.cq[warp];
    if (win.fast) {
      if (below) fused_pass<kVec, true, true>(row, V, win, k, vk, cnt, q, h, f);
      else fused_pass<kVec, true, false>(row, V, win, k, vk, cnt, q, h, f);
    } else {
      if (below) fused_pass<kVec, false, true>(row, V, win, k, vk, cnt, q, h, f);
      else fused_pass<kVec, false, false>(row, V, win, k, vk, cnt, q, h, f);
    }
    __syncthreads();
    M = block_max_f32(fmaxf(__low2float(h), __high2float(h)), ts);
    const float mk = __fmul_rn(M, k);
    if (!isfinite(M)) {
      bad = done = true;
    } else if (key16(__float_as_uint(M) >> 16) <= top) {
      // the window holds the max: its counts serve the search's first windows
      unsigned long long rest = 0, massb = 0;   // mass under the window; of a second window (none at this width)
      if (below) {
        // per thread from the window's lowest value to the max (a factor at most 1), then fixed point
        rest = block_sum_u64(__float2ull_rn(__fmul_rn(f, ex2(vk - mk)) * kMassUnit), ts);
      }
      if (!dok && !dop) {
        kept = bins_mass(cnt, top, k, mk, ts) + massb + rest;
      } else {
        int cur = 0;                        // which count array the last window is in
        bool pre = true;                    // the fused counts are still there
        uint32_t nxt = 0;                   // the next window's top after the last counted one
        trunc_search(
            ts,
            [&](uint32_t hi, bool blw) -> unsigned long long {
              if (pre && hi == top) { cur = 0; nxt = hi - 256u; return blw ? massb + rest : 0ull; }
              pre = false;
              cur = 0;
              return trunc_window<kVec>(row, V, hi, blw, k, mk, ts, nxt);
            },
            [&](int d) { return ts.cnt[cur][d]; }, [&](uint32_t) { return nxt; }, top, topk, topp, dok, dop, k,
            mk, kmin, kept);
      }
      done = true;
    }
  }
  if (!done) {
    // the estimate missed (or no window fits): the max, then windows from it down
    if (!fused) {
      __nv_bfloat162 h = __floats2bfloat162_rn(-INFINITY, -INFINITY);
      for_each_vec<kVec>(row, V, [&](const uint4& v, int) {
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
        h = __hmax2(h, __hmax2(__hmax2(p2[0], p2[1]), __hmax2(p2[2], p2[3])));
      });
      M = block_max_f32(fmaxf(__low2float(h), __high2float(h)), ts);
    }
    bad = !isfinite(M);
    const float mk = __fmul_rn(M, k);
    const uint32_t ktop = key16(__float_as_uint(M) >> 16);
    if (bad) {
    } else if (!dok && !dop) {
      kept = trunc_total<kVec>(row, V, k, mk, ts);
    } else {
      uint32_t nxt = 0;
      trunc_search(
          ts, [&](uint32_t hi, bool below) { return trunc_window<kVec>(row, V, hi, below, k, mk, ts, nxt); },
          [&](int d) { return ts.cnt[0][d]; }, [&](uint32_t) { return nxt; }, ktop, topk, topp, dok, dop, k, mk,
          kmin, kept);
    }
  }
  const float mk = __fmul_rn(M, k);
  if (tid == 0) {
    RowInfo r;
    r.mk = mk;
    // a row without a distribution is marked by invs = 0 (otherwise invs is in (0, 1]) and
    // keeps nothing
    r.invs = bad ? 0.f : __frcp_rn(float(double(kept) / double(kMassUnit)));
    r.tau = bad ? INFINITY : (kmin == 0 ? -INFINITY : key16_value(kmin));
    r.arg = 0;
    *out = r;
  }
}

// One warp: sequence b's acceptance decisions on the truncated p', q' (or the greedy compare)
// and the plan of its draw (returned in lane 0).  `writer`: also the diag entries and, for a
// greedy sequence, its outputs (one warp per sequence does that).
__device__ PlanRec trunc_decide(const Args& a, const RowInfo* info, int nslots, int b, bool writer) {
  const int lane = int(threadIdx.x) & 31;
  const Seq<Bf16, true> sq(a, b);
  const int g = sq.g, gmax = a.gmax;
  const RowInfo* ri = info + int64_t(b) * nslots;
  bool acc = false, valid = false;
  float p = NAN, q = NAN;
  // the rows' records, loaded with the draft ids: lane i holds target row i and draft row i,
  // lane g (lane 0 when g = 32) the bonus row's invs
  RowInfo rp = {0.f, 1.f, 0.f, 0}, rq = {0.f, 1.f, 0.f, 0};
  float binvs = 1.f;
  if (sq.sampling) {
    if (lane < g) {
      rp = ri[lane];
      rq = ri[gmax + 1 + lane];
    }
    if (lane == (g & 31)) binvs = ri[g].invs;
  }
  if (lane < g) {
    const int d = __ldg(&a.draft_tokens[int64_t(b) * gmax + lane]);
    valid = d >= 0 && int64_t(d) < a.V;
    if (valid) {
      if (sq.sampling) {
        const float xp = Bf16::at(target_row<Bf16>(a, b, lane), d);
        const float xq = Bf16::at(static_cast<const uint16_t*>(a.draft) + (int64_t(b) * gmax + lane) * a.V, d);
        p = xp >= rp.tau ? prob(xp, sq.k, rp.mk, rp.invs) : 0.f;
        q = xq >= rq.tau ? prob(xq, sq.k, rq.mk, rq.invs) : 0.f;
        const float u = __ldg(&a.u_accept[int64_t(b) * gmax + lane]);
        acc = (p == 0.f) ? (u < 0.f) : (p >= q ? (u < 1.f) : (__fmul_rn(u, q) < p));
      } else {
        acc = d == ri[lane].arg;
      }
    }
  }
  const unsigned keep = __ballot_sync(kFull, acc);
  const unsigned rej = ~keep & (g >= 32 ? kFull : ((1u << g) - 1u));
  const int m = rej ? __ffs(rej) - 1 : g;
  const unsigned bad = __ballot_sync(kFull, lane < g && !valid);
  int flags = sq.flags;
  if (m < g && ((bad >> m) & 1u)) flags |= SPEC_ST_BAD_DRAFT;
  // a row without a distribution (its record's invs is 0): target rows 0..g, draft rows 0..g-1
  if (__any_sync(kFull, !(rp.invs > 0.f) || !(rq.invs > 0.f) || !(binvs > 0.f))) flags |= SPEC_ST_BAD_ROW;
  if (writer && a.diag) {   // gmax <= 32: lane i writes draft i's p'(d_i), q'(d_i)
    float* dg = a.diag + int64_t(b) * (2 * gmax + 1);
    if (lane < gmax) {
      dg[2 * lane] = (sq.sampling && lane < g) ? p : NAN;
      dg[2 * lane + 1] = (sq.sampling && lane < g) ? q : NAN;
    }
    if (!sq.sampling && lane == 0) dg[2 * gmax] = NAN;
  }
  PlanRec pr = {};
  if (!sq.sampling) {
    if (!writer) return pr;
    // the round's commit, when the call carries one (lane 0), then the outputs and their
    // history copies
    int hist = -1, cf = 0;
    if (lane == 0) cf = commit_apply(a, b, m, commit_load(a, b), &hist);
    hist = __shfl_sync(kFull, hist, 0);
    for (int i = lane; i <= gmax; i += 32) {
      int v = -1;
      if (i < m) v = a.draft_tokens[int64_t(b) * gmax + i];
      else if (i == m) v = ri[m].arg;
      put_output(a, b, i, m, v, hist);
    }
    if (lane == 0) {
      a.num_accepted[b] = m;
      if (a.status) a.status[b] = flags | cf;
    }
    return pr;
  }
  if (lane == 0) {
    const RowInfo rp = ri[m];
    pr.m = m;
    pr.g = g;
    pr.flags = flags;
    pr.pair = m < g ? 1 : 0;
    pr.mkp = rp.mk;
    pr.invp = rp.invs;
    pr.taup = rp.tau;
    if (pr.pair) {
      const RowInfo rq = ri[gmax + 1 + m];
      pr.mkq = rq.mk;
      pr.invq = rq.invs;
      pr.tauq = rq.tau;
    } else {
      pr.mkq = pr.invq = 0.f;
      pr.tauq = 0.f;
    }
  }
  return pr;
}

// Draw chunk dc of sequence b (sampling sequences): warp 0 first takes the sequence's decisions
// (every chunk alike, so no plan is handed over; chunk 0 also writes the diag and a greedy
// sequence's outputs), then the chunk's part of the draw; the last chunk to finish selects the
// token and writes the outputs.
template <bool kVec>
__global__ void __launch_bounds__(kThreads, kVec ? kMinBlocks : 1) trunc_draw_kernel(const Args a, const Geo geo, const Work w,
                                                              RowInfo* info, int nslots) {
  __shared__ Shared sm;
  const int64_t idx = int64_t(blockIdx.x);
  const int dc = int(idx % geo.DCL), b = int(idx / geo.DCL);
  const Seq<Bf16, true> sq(a, b);
  if (!sq.sampling && dc != 0) return;
  // launched while the row kernel finishes: its records are complete and visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x < 32) {
    const PlanRec pr = trunc_decide(a, info, nslots, b, dc == 0);
    if (threadIdx.x == 0) sm.plan = pr;
  }
  __syncthreads();
  if (sq.sampling) {
    const PlanRec pl = sm.plan;
    draw_chunk<Bf16, kVec, true, true>(a, geo, w, sq, pl, dc, sm);
  } else {
    sm.last = true;   // unit 0 of a greedy sequence clears what the call used
  }
  __syncthreads();
  if (!sm.last) return;
  // the selector (or a greedy sequence's unit 0), after every chunk of b has read its rows'
  // records: they return to zero
  for (int i = int(threadIdx.x); i < nslots; i += kThreads) info[int64_t(b) * nslots + i] = RowInfo{0.f, 0.f, 0.f, 0};
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

struct Split {
  int cl, chunk;     // row chunks
  int dcl, dchunk;   // draw chunks
};

// n chunks of len ids (a multiple of `gran`) covering V, about `target` ids each, n <= nmax
void cut(int64_t V, int target, int nmax, int gran, int& n, int& len) {
  int64_t c = (V + target - 1) / target;
  if (c < 1) c = 1;
  if (c > nmax) c = nmax;
  int64_t l = (V + c - 1) / c;
  l = (l + gran - 1) / gran * gran;
  n = int((V + l - 1) / l);
  len = int(l);
}

Split make_split(int64_t V) {
  Split s;
  cut(V, kChunkTarget, kMaxChunks, 8, s.cl, s.chunk);
  // draw chunks split evenly into kWarps sub-ranges of whole 16-byte vectors
  cut(V, kDrawChunkTarget, kMaxDrawChunks, kWarps * 8, s.dcl, s.dchunk);
  return s;
}

size_t align64(size_t x) { return (x + 63) & ~size_t(63); }

// Workspace layout: counters and published words only, all zero between calls (each call
// returns every word it used to zero), so calls of any sizes can share one workspace.
struct WsLayout {
  size_t cnt, bdone, planw, state, part, xd, mass, info, end;
};

WsLayout ws_layout(int B, int gmax, int64_t V) {
  const Split s = make_split(V);
  const size_t nslots = size_t(2 * gmax + 1);
  WsLayout L;
  L.cnt = 0;
  L.bdone = L.cnt + align64(size_t(B) * 4);
  L.planw = L.bdone + align64(size_t(B) * 4);
  L.state = L.planw + align64(size_t(B) * 32);
  L.part = L.state + align64(size_t(B) * s.dcl * 4);
  L.xd = L.part + align64(size_t(B) * nslots * s.cl * 8);
  L.mass = L.xd + align64(size_t(B) * nslots * 8);
  L.info = L.mass + align64(size_t(B) * s.dcl * kWarps * 8);   // truncated sampling only
  L.end = L.info + align64(size_t(B) * nslots * sizeof(RowInfo));
  return L;
}

bool ws_fits(int B, int gmax, int64_t V, size_t ws_bytes) { return ws_layout(B, gmax, V).end <= ws_bytes; }

// smallest workspace that fits a call of these sizes (a multiple of 64 bytes)
size_t ws_required(int B, int gmax, int64_t V) {
  const size_t n = ws_layout(B, gmax, V).end;
  return n > 64 ? n : 64;
}

Work ws_views(void* ws, const WsLayout& L) {
  unsigned char* p = static_cast<unsigned char*>(ws);
  Work w;
  w.cnt = reinterpret_cast<int*>(p + L.cnt);
  w.bdone = reinterpret_cast<int*>(p + L.bdone);
  w.planw = reinterpret_cast<uint64_t*>(p + L.planw);
  w.state = reinterpret_cast<int*>(p + L.state);
  w.part = reinterpret_cast<uint64_t*>(p + L.part);
  w.xd = reinterpret_cast<uint64_t*>(p + L.xd);
  w.mass = reinterpret_cast<uint64_t*>(p + L.mass);
  return w;
}

std::mutex g_occ_mu;

template <class E, bool kVec, bool kMixed>
int launch(const Args& args, int dtype, void* ws, size_t ws_bytes, void* stream) {
  auto fn = verify_kernel<E, kVec, kMixed>;
  const Split sp = make_split(args.V);
  if (args.V > (dtype == SPEC_BF16 ? (int64_t(1) << 21) : (int64_t(1) << 20))) {
    set_error("V=%lld too large (at most 2^21 bf16 or 2^20 fp32 ids)", (long long)args.V);
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
  const WsLayout L = ws_layout(args.B, args.gmax, args.V);
  Geo geo;
  geo.CL = sp.cl;
  geo.chunk = sp.chunk;
  geo.DCL = sp.dcl;
  geo.dchunk = sp.dchunk;
  geo.nslots = kMixed ? 2 * args.gmax + 1 : args.gmax + 1;   // greedy-only reads no draft rows
  const int brows = kMixed ? (geo.DCL + geo.CL - 1) / geo.CL : 0;   // grid rows of B units
  const int G = geo.CL * (geo.nslots + brows);                       // units per group
  // B units of a sequence come about kDrawWaves waves of resident blocks after its A units
  const size_t dyn_smem = 0;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  {
    static int cached[64] = {};
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (dev < 64 && cached[dev]) {
      per_sm = cached[dev];
    } else {
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
  if (geo.delta > kMaxGroups / 4) geo.delta = kMaxGroups / 4;
  // sequences whose draws wait for the end: about as many as kDeferBytes of draw rows (the
  // HBM the draw tail leaves idle), which miss L2 then but fill that idle time
  const int64_t draw_row_bytes = 2 * args.V * (dtype == SPEC_BF16 ? 2 : 4);
  geo.ndefer = kMixed ? int((kDeferBytes + draw_row_bytes - 1) / draw_row_bytes) : 0;
  if (geo.ndefer > kMaxGroups / 4) geo.ndefer = kMaxGroups / 4;
  const Work w = ws_views(ws, L);
  // one launch covers at most kMaxGroups groups (the grid's z limit); larger batches take
  // several launches over consecutive sequence ranges, each complete on its own
  const int per_launch = kMaxGroups - geo.delta - geo.ndefer;
  for (int b0 = 0; b0 < args.B; b0 += per_launch) {
    geo.b0 = b0;
    geo.b1 = b0 + per_launch < args.B ? b0 + per_launch : args.B;
    const int groups = kMixed ? draw_groups(geo.b1 - b0, geo.delta, geo.ndefer) : geo.b1 - b0;
    const dim3 grid(unsigned(geo.CL), unsigned(geo.nslots + brows), unsigned(groups));
    fn<<<grid, kThreads, dyn_smem, static_cast<cudaStream_t>(stream)>>>(args, geo, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "verify kernel launch");
    count_launch();
  }
  return SPEC_OK;
}

// truncated sampling: thresholds per row, then decisions and the draw per sequence; two launches
template <bool kVec>
int launch_truncated(const Args& args, const TruncArgs& t, void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !ws_fits(args.B, args.gmax, args.V, ws_bytes)) {
    set_error("workspace of %zu bytes is smaller than the %zu bytes needed", ws ? ws_bytes : size_t(0),
              ws_required(args.B, args.gmax, args.V));
    return SPEC_ENOSPACE;
  }
  if (reinterpret_cast<uintptr_t>(ws) % 64 != 0) {
    set_error("workspace must be 64-byte aligned");
    return SPEC_EINVAL;
  }
  const Split sp = make_split(args.V);
  const WsLayout L = ws_layout(args.B, args.gmax, args.V);
  const Work w = ws_views(ws, L);
  unsigned char* base = static_cast<unsigned char*>(ws);
  RowInfo* info = reinterpret_cast<RowInfo*>(base + L.info);
  const int nslots = 2 * args.gmax + 1;
  Geo geo = {};
  geo.CL = sp.cl;
  geo.chunk = sp.chunk;
  // draw chunks of about kTruncDrawChunk ids, no more than the workspace layout holds
  cut(args.V, kTruncDrawChunk, sp.dcl, kWarps * 8, geo.DCL, geo.dchunk);
  geo.nslots = nslots;
  geo.b0 = 0;
  geo.b1 = args.B;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t rows = int64_t(args.B) * nslots;
  trunc_rows_kernel<kVec><<<unsigned(rows), kThreads, 0, s>>>(args, t, info, nslots);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "truncation rows kernel launch");
  count_launch();
  {
    // programmatic dependent launch: the draw's blocks start as the row kernel's drain
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(int64_t(args.B) * geo.DCL));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, trunc_draw_kernel<kVec>, args, geo, w, info, nslots);
  }
  if (e != cudaSuccess) return cuda_fail(e, "truncation draw kernel launch");
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
int dispatch_on(const Args& a, int dtype, void* ws, size_t ws_bytes, void* stream) {
  const bool vec = vec_ok(a.target, dtype, a.V) && vec_ok(a.draft, dtype, a.V) && vec_ok(a.saved, dtype, a.V);
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
  if (B < 0 || gmax < 0 || gmax > SPEC_MAX_TREE_NODES || V < 1 || (dtype != SPEC_BF16 && dtype != SPEC_F32)) return 0;
  return ws_required(B, gmax, V);
}

namespace specverify {
namespace {

// The commit a fused verify-and-commit call carries (kv_target null: none).
struct CommitArgs {
  int32_t* kv_target;
  int32_t* kv_draft;
  int add;
  int32_t* history;
  int32_t* committed_len;
  int cap;
};

// host checks of a fused call's commit arguments, the same as spec_commit_kv_lengths makes
int check_commit(const CommitArgs& c) {
  if (!c.kv_target) {
    set_error("null required pointer (target_kv_len)");
    return SPEC_EINVAL;
  }
  if ((c.history != nullptr) != (c.committed_len != nullptr)) {
    set_error("history and committed_len must be given together");
    return SPEC_EINVAL;
  }
  if (c.history && c.cap < 1) {
    set_error("history capacity %d < 1", c.cap);
    return SPEC_EINVAL;
  }
  return SPEC_OK;
}

void set_commit(Args& a, const CommitArgs* c) {
  if (!c) return;
  a.kv_target = c->kv_target;
  a.kv_draft = c->kv_draft;
  a.kv_add = c->add ? 1 : 0;
  a.history = c->history;
  a.committed_len = c->committed_len;
  a.cap = c->cap;
}

// The verify calls on either layout: saved == null is the one-array layout.
int verify_greedy(const void* saved, const void* target, int dtype, const int32_t* draft_tokens,
                  const int32_t* num_draft, int B, int gmax, int V, int32_t* out_tokens, int32_t* num_accepted,
                  int32_t* status, void* workspace, size_t workspace_bytes, void* stream,
                  const CommitArgs* ck = nullptr) {
  Args a = {};
  set_commit(a, ck);
  a.saved = saved;
  a.target = target;
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

int verify_sample(const void* saved, const void* target, const void* draft_logits, int dtype,
                  const int32_t* draft_tokens, const int32_t* num_draft, const float* temperature,
                  const float* u_accept, const float* u_sample, int B, int gmax, int V, int32_t* out_tokens,
                  int32_t* num_accepted, float* diag, int32_t* status, void* workspace, size_t workspace_bytes,
                  void* stream, const CommitArgs* ck = nullptr) {
  if (!temperature || !u_sample || (gmax > 0 && (!draft_logits || !u_accept))) {
    set_error("null required pointer (draft_logits, temperature, u_accept or u_sample)");
    return SPEC_EINVAL;
  }
  Args a = {};
  set_commit(a, ck);
  a.saved = saved;
  a.target = target;
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

// the split layout's extra check: the block rows are required when there are drafts
int check_block(const void* block, int B, int gmax) {
  if (B > 0 && gmax > 0 && !block) {
    set_error("null required pointer (block_logits)");
    return SPEC_EINVAL;
  }
  return SPEC_OK;
}

}  // namespace
}  // namespace specverify

extern "C" int spec_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens,
                                  const int32_t* num_draft, int B, int gmax, int V,
                                  int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK || B == 0) return rc;
  return verify_greedy(nullptr, target_logits, dtype, draft_tokens, num_draft, B, gmax, V, out_tokens, num_accepted,
                       status, workspace, workspace_bytes, stream);
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
  if (rc != SPEC_OK || B == 0) return rc;
  return verify_sample(nullptr, target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, u_accept,
                       u_sample, B, gmax, V, out_tokens, num_accepted, diag, status, workspace, workspace_bytes,
                       stream);
}

extern "C" int spec_verify_greedy_commit(const void* target_logits, int dtype, const int32_t* draft_tokens,
                                         const int32_t* num_draft, int B, int gmax, int V, int32_t* out_tokens,
                                         int32_t* num_accepted, int32_t* status, void* workspace,
                                         size_t workspace_bytes, int32_t* target_kv_len, int32_t* draft_kv_len,
                                         int correction_processed, int32_t* history, int32_t* committed_len,
                                         int cap, void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK || B == 0) return rc;
  const CommitArgs ck = {target_kv_len, draft_kv_len, correction_processed, history, committed_len, cap};
  rc = check_commit(ck);
  if (rc != SPEC_OK) return rc;
  return verify_greedy(nullptr, target_logits, dtype, draft_tokens, num_draft, B, gmax, V, out_tokens, num_accepted,
                       status, workspace, workspace_bytes, stream, &ck);
}

extern "C" int spec_verify_sample_commit(const void* target_logits, const void* draft_logits, int dtype,
                                         const int32_t* draft_tokens, const int32_t* num_draft,
                                         const float* temperature, const float* u_accept, const float* u_sample,
                                         int B, int gmax, int V, int32_t* out_tokens, int32_t* num_accepted,
                                         float* diag, int32_t* status, void* workspace, size_t workspace_bytes,
                                         int32_t* target_kv_len, int32_t* draft_kv_len, int correction_processed,
                                         int32_t* history, int32_t* committed_len, int cap, void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK || B == 0) return rc;
  const CommitArgs ck = {target_kv_len, draft_kv_len, correction_processed, history, committed_len, cap};
  rc = check_commit(ck);
  if (rc != SPEC_OK) return rc;
  return verify_sample(nullptr, target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, u_accept,
                       u_sample, B, gmax, V, out_tokens, num_accepted, diag, status, workspace, workspace_bytes,
                       stream, &ck);
}

extern "C" int spec_verify_greedy_split(const void* saved_logits, const void* block_logits, int dtype,
                                        const int32_t* draft_tokens, const int32_t* num_draft, int B, int gmax,
                                        int V, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int rc = check_common(saved_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc == SPEC_OK) rc = check_block(block_logits, B, gmax);
  if (rc != SPEC_OK || B == 0) return rc;
  return verify_greedy(saved_logits, block_logits, dtype, draft_tokens, num_draft, B, gmax, V, out_tokens,
                       num_accepted, status, workspace, workspace_bytes, stream);
}

extern "C" int spec_verify_sample_split(const void* saved_logits, const void* block_logits,
                                        const void* draft_logits, int dtype, const int32_t* draft_tokens,
                                        const int32_t* num_draft, const float* temperature,
                                        const float* u_accept, const float* u_sample, int B, int gmax, int V,
                                        int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                        int32_t* status, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int rc = check_common(saved_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc == SPEC_OK) rc = check_block(block_logits, B, gmax);
  if (rc != SPEC_OK || B == 0) return rc;
  return verify_sample(saved_logits, block_logits, draft_logits, dtype, draft_tokens, num_draft, temperature,
                       u_accept, u_sample, B, gmax, V, out_tokens, num_accepted, diag, status, workspace,
                       workspace_bytes, stream);
}

namespace specverify {
namespace {

// The truncated call on either layout: saved == nullptr, target [B][gmax+1][V]; or saved
// [B][V] (row 0) and target [B][gmax][V] (rows 1..gmax).
int verify_truncated(const void* saved, const void* target, const void* draft_logits, int dtype,
                     const int32_t* draft_tokens, const int32_t* num_draft, const float* temperature,
                     const int32_t* top_k, const float* top_p, const float* u_accept, const float* u_sample, int B,
                     int gmax, int V, int32_t* out_tokens, int32_t* num_accepted, float* diag, int32_t* status,
                     void* workspace, size_t workspace_bytes, void* stream, const CommitArgs* ck = nullptr) {
  if (dtype != SPEC_BF16) {
    set_error("truncated sampling takes bf16 logits");
    return SPEC_EDTYPE;
  }
  if (V > (1 << 21)) {
    set_error("V=%d too large (at most 2^21 bf16 ids)", V);
    return SPEC_ENOSPACE;
  }
  if (B == 0) return SPEC_OK;
  if (!temperature || !u_sample || (gmax > 0 && (!draft_logits || !u_accept))) {
    set_error("null required pointer (draft_logits, temperature, u_accept or u_sample)");
    return SPEC_EINVAL;
  }
  Args a = {};
  set_commit(a, ck);
  a.saved = saved;
  a.target = target;
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
  TruncArgs t = {top_k, top_p};
  const bool vec = vec_ok(target, dtype, V) && vec_ok(draft_logits, dtype, V) && vec_ok(saved, dtype, V);
  return vec ? launch_truncated<true>(a, t, workspace, workspace_bytes, stream)
             : launch_truncated<false>(a, t, workspace, workspace_bytes, stream);
}

}  // namespace
}  // namespace specverify

extern "C" int spec_verify_sample_truncated(const void* target_logits, const void* draft_logits, int dtype,
                                            const int32_t* draft_tokens, const int32_t* num_draft,
                                            const float* temperature, const int32_t* top_k, const float* top_p,
                                            const float* u_accept, const float* u_sample, int B, int gmax, int V,
                                            int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                            int32_t* status, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  const int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK) return rc;
  return verify_truncated(nullptr, target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, top_k,
                          top_p, u_accept, u_sample, B, gmax, V, out_tokens, num_accepted, diag, status, workspace,
                          workspace_bytes, stream);
}

extern "C" int spec_verify_sample_truncated_commit(
    const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
    const int32_t* num_draft, const float* temperature, const int32_t* top_k, const float* top_p,
    const float* u_accept, const float* u_sample, int B, int gmax, int V, int32_t* out_tokens, int32_t* num_accepted,
    float* diag, int32_t* status, void* workspace, size_t workspace_bytes, int32_t* target_kv_len,
    int32_t* draft_kv_len, int correction_processed, int32_t* history, int32_t* committed_len, int cap,
    void* stream) {
  clear_error();
  int rc = check_common(target_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc != SPEC_OK || B == 0) return rc;
  const CommitArgs ck = {target_kv_len, draft_kv_len, correction_processed, history, committed_len, cap};
  rc = check_commit(ck);
  if (rc != SPEC_OK) return rc;
  return verify_truncated(nullptr, target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, top_k,
                          top_p, u_accept, u_sample, B, gmax, V, out_tokens, num_accepted, diag, status, workspace,
                          workspace_bytes, stream, &ck);
}

extern "C" int spec_verify_sample_truncated_split(const void* saved_logits, const void* block_logits,
                                                  const void* draft_logits, int dtype, const int32_t* draft_tokens,
                                                  const int32_t* num_draft, const float* temperature,
                                                  const int32_t* top_k, const float* top_p, const float* u_accept,
                                                  const float* u_sample, int B, int gmax, int V, int32_t* out_tokens,
                                                  int32_t* num_accepted, float* diag, int32_t* status,
                                                  void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int rc = check_common(saved_logits, dtype, draft_tokens, B, gmax, V, out_tokens, num_accepted);
  if (rc == SPEC_OK) rc = check_block(block_logits, B, gmax);
  if (rc != SPEC_OK) return rc;
  return verify_truncated(saved_logits, block_logits, draft_logits, dtype, draft_tokens, num_draft, temperature,
                          top_k, top_p, u_accept, u_sample, B, gmax, V, out_tokens, num_accepted, diag, status,
                          workspace, workspace_bytes, stream);
}

namespace specverify {
namespace {
int verify_tree(const void* target_logits, int dtype, const int32_t* node_tokens, const int32_t* node_parents,
                const int32_t* num_nodes, int B, int nmax, int V, int32_t* out_tokens, int32_t* num_accepted,
                int32_t* path_nodes, int32_t* status, void* workspace, size_t workspace_bytes, void* stream,
                const CommitArgs* ck) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) {
    set_error("unknown dtype code %d", dtype);
    return SPEC_EDTYPE;
  }
  if (B < 0 || V < 1 || V > (1 << 30) || nmax < 0) {
    set_error("bad sizes B=%d nmax=%d V=%d", B, nmax, V);
    return SPEC_EINVAL;
  }
  if (nmax > SPEC_MAX_TREE_NODES) {
    set_error("nmax=%d exceeds SPEC_MAX_TREE_NODES=%d", nmax, SPEC_MAX_TREE_NODES);
    return SPEC_ENOSPACE;
  }
  if (B == 0) return SPEC_OK;
  if (!target_logits || !out_tokens || !num_accepted || (nmax > 0 && (!node_tokens || !node_parents))) {
    set_error("null required pointer");
    return SPEC_EINVAL;
  }
  if (ck) {
    const int rc = check_commit(*ck);
    if (rc != SPEC_OK) return rc;
  }
  Args a = {};
  set_commit(a, ck);
  a.target = target_logits;
  a.draft_tokens = node_tokens;
  a.parents = node_parents;
  a.path_nodes = path_nodes;
  a.num_draft = num_nodes;
  a.V = V;
  a.B = B;
  a.gmax = nmax;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.status = status;
  return dispatch_on<false>(a, dtype, workspace, workspace_bytes, stream);
}
}  // namespace
}  // namespace specverify

extern "C" int spec_verify_tree_greedy(const void* target_logits, int dtype, const int32_t* node_tokens,
                                       const int32_t* node_parents, const int32_t* num_nodes, int B, int nmax,
                                       int V, int32_t* out_tokens, int32_t* num_accepted, int32_t* path_nodes,
                                       int32_t* status, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  return verify_tree(target_logits, dtype, node_tokens, node_parents, num_nodes, B, nmax, V, out_tokens,
                     num_accepted, path_nodes, status, workspace, workspace_bytes, stream, nullptr);
}

extern "C" int spec_verify_tree_greedy_commit(const void* target_logits, int dtype, const int32_t* node_tokens,
                                              const int32_t* node_parents, const int32_t* num_nodes, int B,
                                              int nmax, int V, int32_t* out_tokens, int32_t* num_accepted,
                                              int32_t* path_nodes, int32_t* status, void* workspace,
                                              size_t workspace_bytes, int32_t* target_kv_len, int32_t* draft_kv_len,
                                              int correction_processed, int32_t* history, int32_t* committed_len,
                                              int cap, void* stream) {
  clear_error();
  const CommitArgs ck = {target_kv_len, draft_kv_len, correction_processed, history, committed_len, cap};
  return verify_tree(target_logits, dtype, node_tokens, node_parents, num_nodes, B, nmax, V, out_tokens,
                     num_accepted, path_nodes, status, workspace, workspace_bytes, stream, &ck);
}

// ------------------------------------------------------------------------------------------
// spec_verify_sample_static: the same verification with a workspace compiled into the library
// ------------------------------------------------------------------------------------------
//
// For callers that cannot allocate device memory at the point of the call: a serving loop
// whose memory is fixed after start-up, or code between a framework's allocations that must
// not add one.  The workspace is one file-scope device array per device (every call of this
// entry point on that device shares it).  Every call looks its address up with
// cudaGetSymbolAddress (which allocates nothing); the first call on a device, and the first
// after a device reset has reloaded the library's module at a new address, also clears the
// array and waits for that.  Nothing is allocated, by this call or by any routine it calls.

namespace specverify {
namespace {

constexpr size_t kStaticWsBytes = SPEC_STATIC_WORKSPACE_BYTES;
static_assert(kStaticWsBytes % 64 == 0, "static workspace size");

// The shared workspace: all zero before the first call (the first call on a device clears it)
// and after every completed call.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_mu;
void* g_static_ptr[64] = {};   // the address this device's array was last cleared at

// The device address of the current device's array, cleared first when it is new.
int static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    set_error("device %d: the static workspace serves devices 0..63", dev);
    return SPEC_EINVAL;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_ws);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static workspace");
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_ptr[dev] != p) {
    e = cudaMemset(p, 0, kStaticWsBytes);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static workspace");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static workspace");
    g_static_ptr[dev] = p;
  }
  *out = p;
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
