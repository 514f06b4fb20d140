// Commit of one round: KV length rollback and optional token-history append; stops (end
// token, token budget) that cut a round's emit; plus the library's error and launch-count
// bookkeeping.
//
// Follows the tutorial "投机解码教程：从概率保持、KV Cache 回滚到性能盈亏平衡", §5.1-§5.2
// (both caches trimmed to t+m, then t+m+1 once the replacement/bonus token is processed;
// target length == draft length == committed length; nothing after an EOS in the candidate
// block may reach the cache) and §12.3 (EOS, maximum length and the rejection position agree
// with step-by-step decoding), and the commit pseudocode of the "M013" knowledge-base card,
// §06 (§03: an end token or a length limit may end a round early).

#include <climits>
#include <cstdarg>
#include <cstdio>

#include "common.cuh"

namespace specverify {

namespace {
thread_local char g_err[512] = {0};
std::atomic<uint64_t> g_launches{0};

__global__ void commit_kernel(const int32_t* __restrict__ num_accepted, int B,
                              int32_t* __restrict__ target_kv_len, int32_t* __restrict__ draft_kv_len,
                              int add, const int32_t* __restrict__ out_tokens, int gmax,
                              int32_t* __restrict__ history, int32_t* __restrict__ committed_len,
                              int cap, int32_t* __restrict__ status) {
  const int b = int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x);
  if (b >= B) return;
  int m = num_accepted[b];
  m = m < 0 ? 0 : (m > gmax ? gmax : m);
  int n = m + 1;
  if (history) {
    const int32_t* src = out_tokens + int64_t(b) * (gmax + 1);
    // only the emitted tokens: a round cut by a stop leaves -1 after them
    for (int i = 0; i < n; ++i)
      if (src[i] < 0) {
        n = i;
        break;
      }
    const int c = committed_len[b];
    if (c < 0 || c > cap - n) {
      if (status) status[b] |= SPEC_ST_HISTORY_FULL;
      return;
    }
    int32_t* dst = history + int64_t(b) * cap + c;
    for (int i = 0; i < n; ++i) dst[i] = src[i];
    committed_len[b] = c + n;
  }
  target_kv_len[b] += m + add;
  if (draft_kv_len) draft_kv_len[b] += m + add;
}

// One thread per sequence.  The emit out[0..m] ends at its first end token (kept) and holds
// at most max_new[b] tokens; the rest becomes -1 and m becomes (tokens emitted) - 1, at
// least 0.  A sequence whose last emitted token is the end token, or whose budget is used
// up, gets SPEC_ST_STOPPED.
__global__ void stops_kernel(int32_t* __restrict__ out_tokens, int32_t* __restrict__ num_accepted, int B,
                             int gmax, int eos_id, const int32_t* __restrict__ max_new,
                             int32_t* __restrict__ status) {
  const int b = int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x);
  if (b >= B) return;
  int32_t* out = out_tokens + int64_t(b) * (gmax + 1);
  int m = num_accepted[b];
  m = m < 0 ? 0 : (m > gmax ? gmax : m);
  int n = m + 1;
  if (eos_id >= 0)
    for (int i = 0; i < n; ++i)
      if (out[i] == eos_id) {
        n = i + 1;
        break;
      }
  bool stopped = false;
  if (max_new) {
    const int budget = max_new[b];
    if (n > budget) n = budget < 0 ? 0 : budget;
    stopped = n >= budget;
  }
  if (eos_id >= 0 && n >= 1 && out[n - 1] == eos_id) stopped = true;
  for (int i = n; i <= gmax; ++i) out[i] = -1;
  num_accepted[b] = n > 0 ? n - 1 : 0;
  if (stopped && status) status[b] |= SPEC_ST_STOPPED;
}
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

void clear_error() { g_err[0] = 0; }

void count_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace specverify

using namespace specverify;

extern "C" const char* spec_last_error(void) { return g_err; }

extern "C" uint64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int spec_commit_kv_lengths(const int32_t* num_accepted, int B, int32_t* target_kv_len,
                                      int32_t* draft_kv_len, int correction_processed,
                                      const int32_t* out_tokens, int gmax, int32_t* history,
                                      int32_t* committed_len, int cap, int32_t* status,
                                      void* stream) {
  clear_error();
  if (B < 0 || gmax < 0) {
    set_error("bad sizes B=%d gmax=%d", B, gmax);
    return SPEC_EINVAL;
  }
  if (gmax > SPEC_MAX_TREE_NODES) {   // a chain's gmax, or a tree's nmax
    set_error("gmax=%d exceeds SPEC_MAX_TREE_NODES=%d", gmax, SPEC_MAX_TREE_NODES);
    return SPEC_ENOSPACE;
  }
  if (B == 0) return SPEC_OK;   // empty batch: pointers may be null
  if (!num_accepted || !target_kv_len) {
    set_error("null required pointer (num_accepted or target_kv_len)");
    return SPEC_EINVAL;
  }
  const int given = (out_tokens != nullptr) + (history != nullptr) + (committed_len != nullptr);
  if (given != 0 && given != 3) {
    set_error("out_tokens, history and committed_len must be given together");
    return SPEC_EINVAL;
  }
  if (history && cap < 1) {
    set_error("history capacity %d < 1", cap);
    return SPEC_EINVAL;
  }
  if (B == 0) return SPEC_OK;
  const int threads = 256;
  const int blocks = (B + threads - 1) / threads;
  commit_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      num_accepted, B, target_kv_len, draft_kv_len, correction_processed ? 1 : 0, out_tokens, gmax,
      history, committed_len, cap, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "commit kernel launch");
  count_launch();
  return SPEC_OK;
}

extern "C" int spec_apply_stops(int32_t* out_tokens, int32_t* num_accepted, int B, int gmax, int eos_id,
                                const int32_t* max_new, int32_t* status, void* stream) {
  clear_error();
  if (B < 0 || gmax < 0) {
    set_error("bad sizes B=%d gmax=%d", B, gmax);
    return SPEC_EINVAL;
  }
  if (gmax > SPEC_MAX_TREE_NODES) {   // a chain's gmax, or a tree's nmax
    set_error("gmax=%d exceeds SPEC_MAX_TREE_NODES=%d", gmax, SPEC_MAX_TREE_NODES);
    return SPEC_ENOSPACE;
  }
  if (B == 0) return SPEC_OK;   // empty batch: pointers may be null
  if (!out_tokens || !num_accepted) {
    set_error("null required pointer (out_tokens or num_accepted)");
    return SPEC_EINVAL;
  }
  const int threads = 256;
  const int blocks = (B + threads - 1) / threads;
  stops_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(out_tokens, num_accepted, B, gmax,
                                                                           eos_id, max_new, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "stops kernel launch");
  count_launch();
  return SPEC_OK;
}
