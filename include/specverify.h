/*
 * specverify — batched target-side verify-and-commit step of speculative decoding,
 * as CUDA kernels for sm_103a behind a plain C ABI.
 *
 * One round of speculative decoding is "draft proposal -> target block verification ->
 * accept/reject -> commit tokens and repair caches" (tutorial "投机解码教程：从概率保持、
 * KV Cache 回滚到性能盈亏平衡", §2).  This library is the last two stages for a batch of
 * B independent sequences, given the logits the two models already produced.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library allocates
 *    nothing, keeps no state between calls and never synchronises the host: each call
 *    enqueues its work on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *    default stream) and returns.  Results are valid once the stream reaches that point.
 *  - The verify calls take a caller-owned device WORKSPACE of at least
 *    spec_verify_workspace_bytes(B, gmax, V, dtype) bytes, 64-byte aligned, which must be
 *    zero-filled before its first use.  It holds counters and hand-over words only, and every
 *    completed call returns all of it to zero, so one workspace serves any number of
 *    successive calls of any sizes it fits.  Calls that may run at the same time (different
 *    streams) need different workspaces.
 *  - Arrays are row-major and contiguous:
 *        target_logits [B][gmax+1][V]   row i judges draft i; row 0 is the target's saved
 *                                       prediction for the position after the committed
 *                                       context; row num_draft[b] is the bonus row
 *                                       (the alignment table of the tutorial's §4)
 *        draft_logits  [B][gmax][V]     row i is the draft distribution d_i was drawn from
 *        draft_tokens  [B][gmax]        int32
 *        u_accept      [B][gmax]        float32 uniforms in [0,1), one per acceptance test
 *        u_sample      [B]              float32 uniform in [0,1) for the correction/bonus draw
 *        out_tokens    [B][gmax+1]      int32: the m+1 emitted tokens, then -1
 *    Rows past a sequence's num_draft, and the draft rows of a greedy sequence, are never
 *    read (they may hold anything).
 *  - Logits are bf16 (SPEC_BF16, raw 16-bit patterns) or float32 (SPEC_F32).  They must be
 *    finite or -inf, with at least one finite value per read row; NaN or +inf inputs give
 *    unspecified (but memory-safe) results.
 *  - Return value: SPEC_OK, or an spec_status_t for errors found on the host (bad
 *    arguments, CUDA launch failure); spec_last_error() then describes it.  Nothing is
 *    enqueued when a call fails its argument checks.
 *  - Data-dependent problems never fault or trap the GPU: they set bits in the optional
 *    per-sequence status[B] word (see SPEC_ST_*) and a defined fallback is taken.
 *  - Limits: 0 <= B, 0 <= gmax <= SPEC_MAX_GAMMA, 1 <= V <= 2^21 (bf16) or 2^20 (fp32);
 *    a larger V, or a batch needing more than 2^31-1 thread blocks, returns SPEC_ENOSPACE.
 *    B == 0 is a no-op that enqueues nothing and accepts null pointers (empty tensors have
 *    none).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_EINVAL = 1,   /* null required pointer, bad size, misuse */
  SPEC_EDTYPE = 2,   /* unknown dtype code */
  SPEC_ENOSPACE = 3, /* a size exceeds a documented maximum */
  SPEC_ECUDA = 4     /* a CUDA runtime call or kernel launch failed */
} spec_status_t;

typedef enum { SPEC_BF16 = 0, SPEC_F32 = 1 } spec_dtype_t;

#define SPEC_MAX_GAMMA 32
#define SPEC_MAX_TREE_NODES 63

/* per-sequence status bits */
#define SPEC_ST_BAD_DRAFT 1      /* the stopping draft id was outside [0,V): it counted as rejected */
#define SPEC_ST_R_ZERO 2         /* a rejection met residual mass R == 0: the correction was drawn from p_m */
#define SPEC_ST_CLAMPED_GAMMA 4  /* num_draft[b] was outside [0,gmax] and was clamped */
#define SPEC_ST_HISTORY_FULL 8   /* commit: appending would overflow the history; sequence left untouched */
#define SPEC_ST_TIMEOUT 16       /* a bounded device-side wait ran out: outputs of the sequence not
                                    written; zero-fill the workspace before reusing it */
#define SPEC_ST_STOPPED 32       /* stops: the sequence emitted its end token or used up its budget */
#define SPEC_ST_BAD_TREE 64      /* tree: a node's parent index was not below its own; it and its
                                    subtree counted as rejected */
#define SPEC_ST_BAD_ROW 128      /* sampling: a row the call reads has no finite maximum or holds a
                                    NaN (all -inf, a +inf or a NaN logit), so it defines no
                                    distribution; the sequence's outputs are a well-formed step
                                    (drafts 0..m-1, then one id) whose token is not defined */

/*
 * Greedy verification (temperature 0).
 * Tutorial §3.3-§4 and the greedy table of the "M013" knowledge-base card, §03: with
 * g_i = argmax_v target[b][i][v] (lowest id among equal maxima), m_b is the first i <
 * num_draft[b] with draft_tokens[b][i] != g_i, else num_draft[b]; the step emits
 * draft_tokens[b][0..m-1] followed by g_m (the target's replacement on a mismatch, the
 * bonus token when every draft matched, tutorial §5.3).
 *
 *   target_logits  [B][gmax+1][V], dtype `dtype`
 *   draft_tokens   [B][gmax]
 *   num_draft      [B] drafts per sequence, or NULL for gmax everywhere
 *   out_tokens     [B][gmax+1] (written), num_accepted [B] = m (written)
 *   status         [B] or NULL (written: SPEC_ST_* bits)
 *   workspace      device scratch of workspace_bytes bytes (see the conventions above)
 */
int spec_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens,
                       const int32_t* num_draft, int B, int gmax, int V, int32_t* out_tokens,
                       int32_t* num_accepted, int32_t* status, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Sampling verification (tutorial §7.1-§7.3; card §04-§06; "学徒的草稿" part 2, Steps 3-4).
 * For a sequence with temperature T > 0: p_i = softmax(target[b][i]/T) and
 * q_i = softmax(draft[b][i]/T) (the same T on both sides).  Drafts are tested left to right:
 * d_i is kept iff u_accept[b][i] < min(1, p_i(d_i)/q_i(d_i)); m is the first rejected i (or
 * num_draft[b]).  On a rejection the correction is the inverse-CDF draw, in ascending id
 * order, of max(p_m - q_m, 0)/R at u_sample[b]*R (R its total); if R == 0 it is drawn from
 * p_m instead (SPEC_ST_R_ZERO).  On full acceptance the bonus token is the inverse-CDF draw
 * of p at row num_draft[b].  A sequence with T <= 0 (or NaN) is verified greedily exactly
 * as spec_verify_greedy does, and its draft rows are not used.
 *
 *   draft_logits   [B][gmax][V], same dtype as target_logits
 *   temperature    [B] float32
 *   u_accept       [B][gmax] float32, u_sample [B] float32
 *   diag           NULL or [B][2*gmax+1] float32 (written): diag[b][2i] = p_i(d_i),
 *                  diag[b][2i+1] = q_i(d_i) for every i < num_draft[b] (NaN when d_i is out
 *                  of range, for i >= num_draft[b], and for greedy sequences);
 *                  diag[b][2*gmax] = R on a rejection (0 when it underflowed), the total
 *                  mass of p at the bonus row on full acceptance, NaN for greedy sequences.
 *   The other arguments are as for spec_verify_greedy.
 */
int spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const int32_t* num_draft,
                       const float* temperature, const float* u_accept, const float* u_sample,
                       int B, int gmax, int V, int32_t* out_tokens, int32_t* num_accepted,
                       float* diag, int32_t* status, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Sampling verification with top-k / top-p truncation (the "M013" card §10 and the nxmr note:
 * temperature, top-p or any other logits processing that changes the distribution must show
 * in p and q).  Exactly spec_verify_sample, with p_i and q_i replaced by their truncated,
 * renormalised versions, each side truncating its own distribution at T the same way:
 *   top-k (0 < top_k[b] < V) keeps the ids whose logit is >= the k-th largest logit of the
 *     row (ties kept);
 *   top-p (0 < top_p[b] < 1) then keeps, of those, the ids whose logit is >= t*, the largest
 *     logit t whose kept mass at or above t reaches top_p[b] times the top-k-kept mass (ties
 *     at t* kept).
 * Drafts should have been drawn from the truncated q (the proposer truncates too).  Acceptance,
 * the residual max(p' - q', 0) and the bonus draw then use p' and q'; diag reports p'(d_i),
 * q'(d_i) and the truncated residual mass.  top_k or top_p NULL (or a value outside its range)
 * turns that truncation off for the batch (or the sequence); greedy sequences (T <= 0) are
 * verified greedily.  bf16 logits only (SPEC_EDTYPE otherwise).
 *
 * Cost: the thresholds are found exactly, per row, by counting the logits' 16-bit
 * order-preserving keys in windows of 256 keys from the top.  Usually one pass over each row
 * of a sampling sequence: a sample of the row places the window before the pass, which also
 * takes the row's max.  A row whose max lies more than 96 keys above the sample's, or whose
 * threshold lies below the window, is read again, once per further window that holds ids
 * (runs of keys holding none are skipped).  Then come the decisions and the draw: two kernel
 * launches in all, the second a programmatic dependent launch.  The workspace is
 * spec_verify_workspace_bytes(B, gmax, V, dtype) bytes, as for spec_verify_sample.
 */
int spec_verify_sample_truncated(const void* target_logits, const void* draft_logits, int dtype,
                                 const int32_t* draft_tokens, const int32_t* num_draft,
                                 const float* temperature, const int32_t* top_k, const float* top_p,
                                 const float* u_accept, const float* u_sample, int B, int gmax, int V,
                                 int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                 int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify_sample_truncated on the split layout of spec_verify_sample_split: saved_logits
 * [B][V] is target row 0 and block_logits [B][gmax][V] holds rows 1..gmax (NULL allowed only
 * when gmax == 0).  Same results as the one-array call on their concatenation.
 */
int spec_verify_sample_truncated_split(const void* saved_logits, const void* block_logits,
                                       const void* draft_logits, int dtype, const int32_t* draft_tokens,
                                       const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                                       const float* top_p, const float* u_accept, const float* u_sample, int B,
                                       int gmax, int V, int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                       int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Greedy verification of a draft TREE (tutorial §5.3: the target checks every node of the
 * tree in one forward and keeps the longest accepted root-to-leaf path; card §01: a tree
 * follows its own rules).  Nodes 1..n (n = num_nodes[b], NULL: nmax) carry the draft token
 * node_tokens[b][j-1] and hang below node_parents[b][j-1], which must be smaller than j
 * (0 is the root: the position after the committed context).  Target row j is the target's
 * prediction for the position after node j; row 0 is the saved prediction, as in the chain.
 * Node j is accepted iff its parent is and its token is the argmax of the parent's row
 * (lowest id among equal maxima).  The path ends at the deepest accepted node, the lowest
 * index among equal depths; m is its depth.  The step emits the path's tokens and then the
 * argmax of the last path node's row (the target's replacement, or its bonus token at a
 * leaf), and path_nodes lists the path's node indices, so that the caller can keep the
 * cache entries of exactly those nodes (card §06: trimming a length alone does not repair a
 * tree's cache).  A chain tree (node j below j-1) gives spec_verify_greedy's results.
 * The pages give no sampling rule for trees; this call is greedy only.
 *
 *   target_logits  [B][nmax+1][V]
 *   node_tokens    [B][nmax] int32, node_parents [B][nmax] int32, num_nodes [B] or NULL
 *   out_tokens     [B][nmax+1] (written): the m+1 emitted tokens, then -1
 *   num_accepted   [B] = m (written); path_nodes [B][nmax] or NULL (written): the path's
 *                  node indices in root-to-leaf order, then -1
 *   status         [B] or NULL: SPEC_ST_BAD_TREE, SPEC_ST_BAD_DRAFT (a candidate id outside
 *                  [0,V)), SPEC_ST_CLAMPED_GAMMA (num_nodes outside [0,nmax])
 *   workspace      at least spec_verify_workspace_bytes(B, nmax, V, dtype) bytes
 * Limits: 0 <= nmax <= SPEC_MAX_TREE_NODES (else SPEC_ENOSPACE).
 */
int spec_verify_tree_greedy(const void* target_logits, int dtype, const int32_t* node_tokens,
                            const int32_t* node_parents, const int32_t* num_nodes, int B, int nmax, int V,
                            int32_t* out_tokens, int32_t* num_accepted, int32_t* path_nodes,
                            int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify_tree_greedy followed by spec_commit_kv_lengths (gmax = nmax), fused: the thread
 * that writes a tree's outputs advances its lengths by the accepted path's m (+1) and appends the
 * path's tokens to the history.  The cache entries of the nodes off the path are the caller's to
 * drop (path_nodes lists the kept ones; card §06: trimming a length alone does not repair a
 * tree's cache).  Commit arguments and return values as for spec_verify_sample_commit.
 */
int spec_verify_tree_greedy_commit(const void* target_logits, int dtype, const int32_t* node_tokens,
                                   const int32_t* node_parents, const int32_t* num_nodes, int B, int nmax, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, int32_t* path_nodes,
                                   int32_t* status, void* workspace, size_t workspace_bytes,
                                   int32_t* target_kv_len, int32_t* draft_kv_len, int correction_processed,
                                   int32_t* history, int32_t* committed_len, int cap, void* stream);

/*
 * Both verify calls on the split layout of the target's logits, for engines that keep the
 * prediction saved from the last round apart from the logits of the new block, so that they
 * need not copy the two into one array first.  In the alignment table of the tutorial's §4,
 * row 0 (the target's prediction for the position after the committed context) was produced
 * by the previous round's forward and saved; rows 1..gmax come from this round's forward over
 * the drafts.  The results are exactly those of spec_verify_greedy / spec_verify_sample on the
 * concatenated array target[b] = [saved_logits[b], block_logits[b][0..gmax-1]]:
 *   saved_logits   [B][V]        target row 0 of every sequence
 *   block_logits   [B][gmax][V]  target rows 1..gmax (may be NULL when gmax == 0)
 * The other arguments, the workspace and the status bits are as for those calls.  The 128-bit
 * load path needs every logits array 16-byte aligned with V * element size a multiple of 16;
 * otherwise a scalar path computes the same results.
 */
int spec_verify_greedy_split(const void* saved_logits, const void* block_logits, int dtype,
                             const int32_t* draft_tokens, const int32_t* num_draft, int B, int gmax,
                             int V, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                             void* workspace, size_t workspace_bytes, void* stream);
int spec_verify_sample_split(const void* saved_logits, const void* block_logits,
                             const void* draft_logits, int dtype, const int32_t* draft_tokens,
                             const int32_t* num_draft, const float* temperature,
                             const float* u_accept, const float* u_sample, int B, int gmax, int V,
                             int32_t* out_tokens, int32_t* num_accepted, float* diag,
                             int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify_sample without a caller-owned workspace.  The pages have no counterpart: this
 * is a convenience of this library for callers that cannot allocate device memory where they
 * verify (a serving loop whose memory is fixed after start-up, or a step between a
 * framework's allocations that must not add one).  It computes exactly what
 * spec_verify_sample computes, with the same arguments minus the workspace.
 *
 * The workspace is an array of SPEC_STATIC_WORKSPACE_BYTES bytes compiled into the library,
 * one per device, shared by every call of this function on that device:
 *   - Calls whose sizes need more (spec_verify_workspace_bytes(B, gmax, V, dtype) above
 *     SPEC_STATIC_WORKSPACE_BYTES: B = 1110 at gmax = 4, V = 128256 and B = 910 at
 *     gmax = 4, V = 151936 are the largest that fit) return SPEC_ENOSPACE before touching
 *     the device.
 *   - Every call looks the array's device address up (cudaGetSymbolAddress, which allocates
 *     nothing).  The first call on a device, and the first after a device reset (which
 *     reloads the library's code, possibly at another address), also clears the array and
 *     waits for the clear, so its counters start at zero; make that call outside any stream
 *     capture.  Other calls only launch the kernel.
 *   - Like any workspace, the array is all zero between calls.
 *   - Calls that may overlap (different streams, or threads without ordering) race on the one
 *     array: serialise them, e.g. on one stream.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define SPEC_STATIC_WORKSPACE_BYTES ((size_t)1 << 20)
int spec_verify_sample_static(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_tokens, const int32_t* num_draft,
                              const float* temperature, const float* u_accept,
                              const float* u_sample, int B, int gmax, int V, int32_t* out_tokens,
                              int32_t* num_accepted, float* diag, int32_t* status, void* stream);

/*
 * Bytes of workspace a verify call with these sizes needs (any verify entry point; pass nmax
 * as gmax for a tree call); 0 for invalid sizes.  Host-only.
 */
size_t spec_verify_workspace_bytes(int B, int gmax, int V, int dtype);

/*
 * Commit one round and roll the KV lengths back (tutorial §5.1-§5.2; card §06).
 * The caches are trimmed to t + m (the accepted prefix of the block the verifier wrote);
 * after the correction or bonus token has been fed through both models they hold
 * t + m + 1.  So, per sequence:
 *     target_kv_len[b] += num_accepted[b] + (correction_processed ? 1 : 0)
 * and the same for draft_kv_len when it is not NULL (invariant: target length == draft
 * length == committed length, tutorial §5.1).  When `history` is not NULL, the emitted
 * tokens -- out_tokens[b][0..m] up to its first -1, which only spec_apply_stops leaves
 * there, so normally all m+1 -- are appended to history[b][committed_len[b]...] and
 * committed_len[b] grows by their count; a sequence whose append would pass `cap` is left
 * entirely untouched (lengths included) and flagged SPEC_ST_HISTORY_FULL in status.
 *
 *   num_accepted   [B] int32 (m, as written by a verify call; values are clamped to
 *                  [0, gmax]); gmax may be a tree call's nmax (up to SPEC_MAX_TREE_NODES)
 *   target_kv_len  [B] int32, read and written; draft_kv_len [B] or NULL
 *   out_tokens     [B][gmax+1] int32, history [B][cap] int32, committed_len [B] int32 —
 *                  all three NULL, or all three given (cap >= 1)
 *   status         [B] or NULL: bits are OR-ed in (not cleared)
 */
int spec_commit_kv_lengths(const int32_t* num_accepted, int B, int32_t* target_kv_len,
                           int32_t* draft_kv_len, int correction_processed,
                           const int32_t* out_tokens, int gmax, int32_t* history,
                           int32_t* committed_len, int cap, int32_t* status, void* stream);

/*
 * Verification and the commit of the same round in one launch: spec_verify_greedy /
 * spec_verify_sample followed by spec_commit_kv_lengths (with that call's out_tokens, gmax
 * and status), fused.  The tutorial's §13.2 asks for the round's decision to stay on the GPU
 * and for small kernels to be merged; here the thread that writes a sequence's outputs also
 * rolls its KV lengths back (tutorial §5.1-§5.2; card §06), so a round costs one launch.
 * Every output -- out_tokens, num_accepted, diag, status, the lengths, history and
 * committed_len -- equals what the two separate calls leave, except that status carries
 * SPEC_ST_HISTORY_FULL in the same word the verify call writes (the separate commit ORs it
 * into the word the verify call wrote: the same value).
 *
 *   target_kv_len  [B] int32, required, read and written; draft_kv_len [B] or NULL
 *   history [B][cap] and committed_len [B]: both NULL, or both given with cap >= 1
 *
 * Returns what the verify call returns, or SPEC_EINVAL for bad commit arguments (nothing is
 * enqueued then).  Use a stops pass (spec_apply_stops) with the separate calls instead:
 * the fused call commits every emitted token.
 */
int spec_verify_greedy_commit(const void* target_logits, int dtype, const int32_t* draft_tokens,
                              const int32_t* num_draft, int B, int gmax, int V, int32_t* out_tokens,
                              int32_t* num_accepted, int32_t* status, void* workspace, size_t workspace_bytes,
                              int32_t* target_kv_len, int32_t* draft_kv_len, int correction_processed,
                              int32_t* history, int32_t* committed_len, int cap, void* stream);
int spec_verify_sample_commit(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_tokens, const int32_t* num_draft,
                              const float* temperature, const float* u_accept, const float* u_sample,
                              int B, int gmax, int V, int32_t* out_tokens, int32_t* num_accepted,
                              float* diag, int32_t* status, void* workspace, size_t workspace_bytes,
                              int32_t* target_kv_len, int32_t* draft_kv_len, int correction_processed,
                              int32_t* history, int32_t* committed_len, int cap, void* stream);

/*
 * spec_verify_sample_truncated followed by spec_commit_kv_lengths, fused in the same way: the
 * thread that writes a sequence's outputs (the selector for a sampling sequence, the decision
 * warp for a greedy one) commits it.  Same arguments as spec_verify_sample_truncated, then
 * the commit's as for spec_verify_sample_commit; same outputs as the two separate calls.
 */
int spec_verify_sample_truncated_commit(const void* target_logits, const void* draft_logits, int dtype,
                                        const int32_t* draft_tokens, const int32_t* num_draft,
                                        const float* temperature, const int32_t* top_k, const float* top_p,
                                        const float* u_accept, const float* u_sample, int B, int gmax, int V,
                                        int32_t* out_tokens, int32_t* num_accepted, float* diag,
                                        int32_t* status, void* workspace, size_t workspace_bytes,
                                        int32_t* target_kv_len, int32_t* draft_kv_len, int correction_processed,
                                        int32_t* history, int32_t* committed_len, int cap, void* stream);

/*
 * Stops: cut each round's emit where step-by-step decoding would have stopped (tutorial
 * §5.2: nothing after an EOS in the candidate block may reach the cache; §12.3: EOS,
 * maximum length and the rejection position must agree with step-by-step decoding; card §03:
 * an end token or a length limit may end a round early).  Run it between a verify call and
 * spec_commit_kv_lengths, on the same stream.
 *
 * Per sequence, the emit out_tokens[b][0..m] (m = num_accepted[b], clamped to [0, gmax];
 * gmax up to SPEC_MAX_TREE_NODES, so a tree call's emit can be cut too)
 * ends at its first token equal to eos_id (kept; eos_id < 0: no end token) and holds at most
 * max_new[b] tokens (the sequence's remaining budget; <= 0 emits nothing; max_new NULL: no
 * budget).  The tokens after the cut become -1 and num_accepted[b] becomes (tokens
 * emitted) - 1, at least 0: every emitted token but the last keeps its cache entries, the
 * last is fed next, as a correction token is.  status[b] (if not NULL) gets
 * SPEC_ST_STOPPED when the last emitted token is eos_id or the budget is used up; such a
 * sequence must not be continued (do not feed its last token).
 *
 *   out_tokens     [B][gmax+1] int32, read and written
 *   num_accepted   [B] int32, read and written
 *   max_new        [B] int32 or NULL
 */
int spec_apply_stops(int32_t* out_tokens, int32_t* num_accepted, int B, int gmax, int eos_id,
                     const int32_t* max_new, int32_t* status, void* stream);

/* Message for the calling thread's last non-OK return ("" if none). */
const char* spec_last_error(void);

/* Kernels this library has launched in this process (all threads, all devices). */
uint64_t spec_launch_count(void);

/*
 * How a verify call splits the vocabulary for this V and dtype: every row is cut into
 * *ctas_per_seq chunks of *chunk ids (the last one ragged), each streamed by one thread
 * block.  Host-only; returns SPEC_OK or SPEC_EINVAL.
 */
int spec_verify_plan(int V, int dtype, int* ctas_per_seq, int* chunk);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
