/* dh.h - C ABI of the GB300 (sm_103a) two-stage draft LM head and greedy draft-tree acceptance.
 *
 * The method (EAGLE-4 summary page, yuxiaoba.github.io/tech/en/eagle-4, section "Retrieve
 * vocabulary candidates cheaply, then score them exactly"): a low-rank head over the full
 * vocabulary retrieves K candidates per row, and only those candidates are scored exactly with the
 * original full-rank head.  Greedy acceptance (daily.dev "EAGLE-4 speeds up LLM inference with an
 * adaptive speculative decoding drafter", section "How it works"): the target scores every drafted
 * node in one pass, drafted tokens are kept while they equal the target's choice and the first
 * mismatch is replaced by the target's own token.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named as device pointers must point to device memory of the current CUDA device; the
 *   caller owns every buffer.  The library allocates no device memory and keeps no per-call state
 *   outside the caller's workspace.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every call is
 *   asynchronous on that stream: it returns after queuing its kernels and never synchronizes.
 * - Arguments are validated on the host before anything is queued.  A rejected call returns a
 *   non-zero dh_status and queues nothing.  A launch failure returns DH_ERR_CUDA.
 * - Bad data that only the device can see (an index out of range, a parent array that is not a
 *   tree) is reported in the outputs as documented per call; the kernels never trap.
 * - dtype: DH_F32 (IEEE binary32) or DH_BF16 (bfloat16, stored as 16-bit words).  Arithmetic is
 *   fp32 with fp32 accumulation for both.
 * - Alignment: every tensor base pointer must be 16-byte aligned, and row lengths in bytes must be
 *   multiples of 16 (bf16: d, r, vocab multiples of 8; fp32: multiples of 4).  Otherwise
 *   DH_ERR_UNSUPPORTED.
 * - Layouts are dense row-major with no padding between rows.
 * - Workspace: caller-provided device memory of at least the size the matching *_workspace query
 *   returns for the same arguments, 256-byte aligned.  Before its first use the workspace must be
 *   zero-filled (for example with cudaMemset); every completed call leaves it ready for the next
 *   call with the same or smaller arguments.  Calls that share a workspace must not overlap in
 *   time (queue them on one stream).
 */
#ifndef DH_H
#define DH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DH_OK = 0,
  DH_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, K outside [1, min(vocab, 1024)] */
  DH_ERR_UNSUPPORTED = 2, /* alignment, dtype or a size above the documented limits          */
  DH_ERR_WORKSPACE = 3,   /* workspace missing, too small or not 256-byte aligned            */
  DH_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed                      */
  DH_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (see dh_workspace_status)     */
  DH_ERR_BAD_INPUT = 6    /* per-row code written to err_out by dh_tree_accept                */
} dh_status;

typedef enum { DH_F32 = 0, DH_BF16 = 1 } dh_dtype;

/* Limits checked on the host. */
#define DH_MAX_K 1024
#define DH_MAX_RANK 1024
#define DH_MAX_VOCAB (1 << 21)
#define DH_MAX_TREE_NODES 1024

/* Human-readable name of a status code (static string, never NULL). */
const char* dh_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
int dh_version(void);

/* Description of the last CUDA failure behind a DH_ERR_CUDA returned to the calling thread
 * ("" if none).  The string is owned by the library and overwritten by the next failure. */
const char* dh_last_error(void);

/* ---------------------------------------------------------------------------------------------
 * Stage 1: low-rank candidate retrieval.
 *
 * EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly"
 * (the low-rank head selects candidates; its scores are not final probabilities); AlphaSignal
 * "EAGLE-4 Triples Qwen3 Inference Speed by Adapting to Serving Load", section "Runtime-sized
 * speculation" (low-rank candidate head: token prediction factored into smaller matrices).
 *
 * For every row b:
 *   t[b,:]   = h[b,:] U                 (fp32 accumulation, then rounded to `dtype`, RNE)
 *   s[b,v]   = t[b,:] V[:,v]            (fp32 accumulation) for every v in [0, vocab)
 *   idx[b,:] = the K vocabulary ids with the largest s[b,v], ordered by (s desc, id asc)
 *   score[b,k] = s[b, idx[b,k]]
 * The B x vocab score matrix is never written to memory.
 *
 * h [B x d], U [d x r], V [r x vocab]: device, `dtype`.
 * idx_out [B x K] int32, score_out [B x K] fp32: device.
 * B = 0 is a no-op.  Limits: r <= DH_MAX_RANK, vocab <= DH_MAX_VOCAB, K <= min(vocab, DH_MAX_K).
 *
 * Precision of t on the small-batch path (bf16 with B <= 4, fp32 with B <= 8, r a multiple of 16):
 * the projection is split over G <= 3 x (SM count) slices of d, each slice summed in fp32 and then
 * added exactly as a 64-bit fixed-point number with 32 fraction bits, so t is bit-identical from
 * call to call.  Range: every slice's partial sum and every |t[b,j]| must stay below 2^31; a slice
 * beyond it raises bit (1 << DH_ERR_UNSUPPORTED) in the workspace status word (dh_workspace_status)
 * and the call's outputs are unspecified.  Resolution: the fixed-point step adds at most G x 2^-33
 * absolute error (under 1e-7 on a GB300) before t is rounded to `dtype`.
 * ------------------------------------------------------------------------------------------- */
size_t dh_lowrank_topk_workspace(int B, int d, int r, int vocab, int K, int dtype);
int dh_lowrank_topk(const void* h, const void* U, const void* V, int B, int d, int r, int vocab,
                    int K, int dtype, int32_t* idx_out, float* score_out, void* workspace,
                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Stage 2: exact rescoring of the candidates with the full-rank head, and their softmax.
 *
 * EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly"
 * (exact logits of the retrieved candidates from the original full-rank head); the products of
 * these draft probabilities are the benefit estimate of section "Why a draft tree needs a cost
 * model".  The softmax runs over the K candidates of a row at temperature 1.
 *
 *   logits[b,k] = h[b,:] . W[idx[b,k], :]   (fp32 accumulation)
 *   probs[b,k]  = exp(logits[b,k] - m_b) / sum_k' exp(logits[b,k'] - m_b),  m_b = max_k logits[b,k]
 *
 * h [B x d], W [vocab x d]: device, `dtype`.  idx [B x K] int32: device.
 * logits_out [B x K] fp32: device.  probs_out [B x K] fp32: device, may be NULL (no softmax).
 * An index outside [0, vocab) is not dereferenced: its logit is NaN, which makes that row's
 * probabilities NaN.  Limits: d <= 8192, K <= DH_MAX_K.  B = 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
size_t dh_exact_rescore_workspace(int B, int d, int vocab, int K, int dtype);
int dh_exact_rescore(const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                     int dtype, float* logits_out, float* probs_out, void* workspace,
                     size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Both stages in one call: dh_lowrank_topk followed by dh_exact_rescore on its candidates.
 *
 * EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
 * the two stages of the draft head, the low-rank retrieval of K candidates and their exact
 * rescoring, computed as one head.  Outputs and their meaning are exactly those of the two calls:
 * idx_out / score_out as dh_lowrank_topk, logits_out / probs_out as dh_exact_rescore (probs_out
 * may be NULL).  h [B x d], U [d x r], V [r x vocab], W [vocab x d]: device, `dtype`, 16-byte
 * aligned, with d, r and vocab rows a multiple of 16 bytes; d <= 8192; limits and error codes as
 * for the two calls (bit for bit, except that where the two calls would use their bulk-copy
 * rescoring kernel, from 2048 (row, candidate) pairs, probabilities agree to rounding).  When the
 * device runs one thread-block cluster of 16, 8, 4 or 2 CTAs per row for all B rows at once (with 4
 * CTAs, for at most 8192 pairs with K <= 64 and 2048 above: up to 36 rows on a GB300; with 2, for
 * K <= 64: up to 76 rows) and K <= 128, the
 * selection and the rescoring run as one kernel, which removes a kernel boundary from the critical
 * path; on the first call per device the library queries how many such clusters fit (the switch
 * DH_FORCE_HEAD, see dh_set_tuning, runs the two calls' kernels instead, or the cluster kernel
 * whatever K).
 * The workspace (dh_draft_head_workspace bytes, 256-byte aligned, caller-owned) must be zero-filled
 * before its first use and not shared by calls that overlap in time; the library leaves it ready
 * for the next call.
 * ------------------------------------------------------------------------------------------- */
size_t dh_draft_head_workspace(int B, int d, int r, int vocab, int K, int dtype);
int dh_draft_head(const void* h, const void* U, const void* V, const void* W, int B, int d, int r, int vocab,
                  int K, int dtype, int32_t* idx_out, float* score_out, float* logits_out, float* probs_out,
                  void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Expanding frontier nodes of the draft tree.
 *
 * EAGLE-4 summary page, section "Why a draft tree needs a cost model": products of draft
 * probabilities approximate a branch's benefit A, and a branch is worth computing when A over its
 * latency cost C passes a threshold (the page's formula is lost; here a child is kept when
 * A > min_benefit, and the caller supplies min_benefit = threshold x C from its latency table for
 * the batch and width).  AlphaSignal page, section "Runtime-sized speculation": a top-k of 1
 * drafts a chain, larger k a tree.
 *
 * Row b is a frontier node with K candidates: idx[b,:] (token ids, e.g. from dh_lowrank_topk) and
 * their exact probabilities probs[b,:] (e.g. from dh_exact_rescore).
 *   order      = the candidates by (probability desc, token asc, position asc); a NaN probability
 *                ranks below every number
 *   child_token[b,c] = idx[b, order[c]],  c < w
 *   child_prob[b,c]  = fp32(parent_prob[b] * probs[b, order[c]])   (parent_prob NULL: 1)
 *   n_keep[b]  = number of c < w with child_prob[b,c] > min_benefit (a prefix; min_benefit <= 0
 *                with finite probabilities keeps all w)
 * probs, child_prob: fp32; idx, child_token, n_keep: int32; all device.  probs, idx [B x K];
 * parent_prob [B] (may be NULL); child_* [B x w]; n_keep [B] (may be NULL).  1 <= w <= K <= DH_MAX_K.
 * No workspace.  Launched with programmatic dependent launch after a rescoring call on the same
 * stream.  B = 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
int dh_expand_children(const float* probs, const int32_t* idx, const float* parent_prob, int B, int K, int w,
                       float min_benefit, int32_t* child_token, float* child_prob, int32_t* n_keep,
                       void* stream);

/* ---------------------------------------------------------------------------------------------
 * Vocabulary-sharded draft head (tensor-parallel serving).
 *
 * EAGLE-4 summary page, section "Adaptation has not eliminated high-load regressions" (the release
 * serves the target with tensor parallelism over four GPUs), and section "Retrieve vocabulary
 * candidates cheaply, then score them exactly".  The vocabulary is split into P contiguous shards;
 * shard p holds V_p = V[:, o_p : o_p + n_p] (its own contiguous [r x n_p] array) and
 * W_p = W[o_p : o_p + n_p, :].  One step of the head on P shards:
 *   1. every shard: dh_lowrank_topk_shard -> its K best (global id, score) per row
 *   2. exchange the P lists (all-gather: 8 x B x K bytes per shard), then dh_merge_topk -> the K
 *      best of the union, the candidates of dh_lowrank_topk on the whole vocabulary: a global top-K
 *      member is in its shard's top K.  (Scores agree to rounding: where the selection re-scores a
 *      group exactly, its summation order differs from the scores kernel's, and which groups it
 *      re-scores depends on the shard; so ids may differ only between near-equal scores.)
 *   3. every shard: dh_exact_rescore_shard on the merged ids -> the logits of the ids it owns (-inf
 *      elsewhere) and its (max, sum of exp) per row
 *   4. exchange logits and pairs (all-gather: (4 x B x K + 8 x B) bytes per shard), then
 *      dh_combine_softmax -> every candidate's logit from its owner and the softmax over the K
 *      candidates (the unsharded probabilities up to rounding)
 * The exchange itself is the caller's (e.g. NCCL); all buffers are device memory.
 *
 * dh_lowrank_topk_shard: dh_lowrank_topk on V_shard [r x vocab_shard] (same arguments, workspace
 *   from dh_lowrank_topk_workspace with vocab_shard), then idx_out += vocab_offset.  Needs
 *   K <= vocab_shard; vocab_offset >= 0 and vocab_offset + vocab_shard <= DH_MAX_VOCAB.
 * dh_merge_topk: idx_parts int32 / score_parts fp32 [P x B x K] (part p = shard p's output) ->
 *   idx_out int32 / score_out fp32 [B x K], ordered by (score desc, id asc); entries with id < 0
 *   or a NaN score are skipped; a row with fewer than K entries is padded with (-1, -inf).
 *   P x K <= DH_MAX_MERGE_ENTRIES.  No workspace.
 * dh_exact_rescore_shard: idx [B x K] global ids; for the ids in [vocab_offset, vocab_offset +
 *   vocab_shard): logits_out[b,k] = h[b,:] . W_shard[idx - vocab_offset, :] as dh_exact_rescore
 *   computes it; other ids: -inf.  stats_out fp32 [B x 2]: per row the maximum m of its logits and
 *   the sum of exp(logit - m) (m = -inf, sum 0 when the shard owns none).  Workspace:
 *   dh_exact_rescore_shard_workspace bytes, zero-filled before first use, as for dh_exact_rescore.
 * dh_combine_softmax: logits_parts [P x B x K] and stats_parts [P x B x 2] from the P shards ->
 *   logits_out [B x K] (each candidate's owned logit: the maximum over the parts) and probs_out
 *   [B x K] (may be NULL): exp(logit - M) / S with M = max_p m_p, S = sum_p sum_p' exp(m_p - M).
 * ------------------------------------------------------------------------------------------- */
#define DH_MAX_MERGE_ENTRIES 8192
int dh_lowrank_topk_shard(const void* h, const void* U, const void* V_shard, int B, int d, int r, int vocab_shard,
                          int vocab_offset, int K, int dtype, int32_t* idx_out, float* score_out, void* workspace,
                          size_t ws_bytes, void* stream);
int dh_merge_topk(const int32_t* idx_parts, const float* score_parts, int P, int B, int K, int32_t* idx_out,
                  float* score_out, void* stream);
size_t dh_exact_rescore_shard_workspace(int B, int d, int vocab_shard, int K, int dtype);
int dh_exact_rescore_shard(const void* h, const void* W_shard, const int32_t* idx, int B, int d, int vocab_shard,
                           int vocab_offset, int K, int dtype, float* logits_out, float* stats_out, void* workspace,
                           size_t ws_bytes, void* stream);
int dh_combine_softmax(const float* logits_parts, const float* stats_parts, int P, int B, int K, float* logits_out,
                       float* probs_out, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Sizing the next draft level by benefit over latency cost.
 *
 * EAGLE-4 summary page, section "Why a draft tree needs a cost model": products of draft
 * probabilities estimate a branch's benefit A in accepted tokens, latency tables indexed by batch
 * and verification width price another level, and each round decides whether to deepen and how wide
 * to go by comparing A with its cost against a threshold (the page's formula is lost; this is its
 * per-branch reading).  AlphaSignal page, section "Runtime-sized speculation": depth and branching
 * are chosen for the active batch size.
 *
 * Request r's frontier has F nodes with Wc candidate children each (e.g. dh_expand_children's
 * outputs): path probabilities child_prob[r,f,k] and tokens child_token[r,f,k], of which the first
 * n_valid[r,f] are valid (n_valid NULL: all Wc).  With the cost row of the current batch (row i of
 * cost [n_bins x (wmax+1)] for the first i with batch <= bin_batch[i], else the last row):
 *   order      = the valid children by (A desc, f asc, k asc); a NaN probability ranks below every
 *                number
 *   child j of the order is kept while A_j > theta x (cost[j+1] - cost[j])  (fp32: the difference
 *                and the product each rounded once; no fused multiply-add), j < wmax
 *   width_out[r] = the number kept (0: do not deepen)
 *   sel_parent[r,j], sel_token[r,j], sel_prob[r,j] = f, token and A of kept child j; -1, -1, 0 for
 *                j >= width (the next frontier, in order)
 * All pointers device; child_* [R x F x Wc], n_valid [R x F], cost fp32, bin_batch int32 [n_bins]
 * (ascending), outputs [R] and [R x wmax].  Limits: F x Wc <= DH_MAX_LEVEL_CHILDREN, wmax <= DH_MAX_K.
 * No workspace.  Launched with programmatic dependent launch after an expansion on the same stream.
 * R = 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
#define DH_MAX_LEVEL_CHILDREN 8192
int dh_size_level(const float* child_prob, const int32_t* child_token, const int32_t* n_valid, int R, int F, int Wc,
                  const float* cost, const int32_t* bin_batch, int n_bins, int wmax, int batch, float theta,
                  int32_t* width_out, int32_t* sel_parent, int32_t* sel_token, float* sel_prob, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Greedy draft-tree acceptance.
 *
 * daily.dev "EAGLE-4 speeds up LLM inference ...", section "How it works"; EAGLE-4 summary page,
 * section "Distribution preservation has algorithmic and implementation conditions" (greedy
 * decoding follows the target's choices); AlphaSignal page, section "Runtime-sized speculation"
 * (top-k = 1 drafts a chain, larger k a tree).
 *
 * Node 0 of each request is the root (the last verified token; its token is ignored).  For node n
 * the target's next-token logits after n are logits[b, n, :].
 *   a[b,n]   = argmax_v logits[b,n,v]                      (ties -> lowest v, exact compare; a NaN
 *              ranks below every number, and a row holding only NaN gives 0)
 *   acc[0]   = 1;  acc[n] = acc[parent[n]] && token[n] == a[b, parent[n]]
 *   last     = the accepted node of greatest depth          (ties -> lowest node index)
 *   len[b]   = depth(last) = number of accepted draft tokens
 *   path[b,:]= root .. last (len+1 node indices, root first), then -1
 *   bonus[b] = a[b, last]   (the target's own token after the accepted path)
 *
 * logits [B x N x vocab]: device, `dtype`.  parent, token [B x N] int32: device; parent[0] = -1 and
 * 0 <= parent[n] < n for n >= 1.
 * argmax_out [B x N] int32 (may be NULL), path_out [B x N] int32, len_out [B] int32,
 * bonus_out [B] int32, err_out [B] int32 (may be NULL): device.
 * A request whose parent array breaks the rule gets len = -1, bonus = -1, an all -1 path and
 * err = DH_ERR_BAD_INPUT (err = 0 otherwise).  N <= DH_MAX_TREE_NODES.  B = 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
size_t dh_tree_accept_workspace(int B, int N, int vocab);
int dh_tree_accept(const void* logits, const int32_t* parent, const int32_t* token, int B, int N,
                   int vocab, int dtype, int32_t* argmax_out, int32_t* path_out, int32_t* len_out,
                   int32_t* bonus_out, int32_t* err_out, void* workspace, size_t ws_bytes,
                   void* stream);

/* ---------------------------------------------------------------------------------------------
 * Chain verification at positive temperature (speculative sampling).
 *
 * EAGLE-4 summary page, section "Distribution preservation has algorithmic and implementation
 * conditions": at positive temperature the target verifies the drafted tokens and a rejection
 * correction keeps the target's distribution; each round's depth is fixed before the round.  For a
 * chain of L drafted tokens that is standard speculative sampling (Leviathan, Kalman and Matias
 * 2023; Chen et al. 2023).  For request b, with target logit rows l_0..l_L (row i: the target's
 * next-token logits after the prefix and the drafted x_0..x_{i-1}) and temperature T:
 *   p_i(v)  = exp(l_i(v)/T - max) / sum_v' exp(l_i(v')/T - max)
 *   q_i(v)  = sum of cand_prob[b,i,k] over the k with cand_idx[b,i,k] = v (0 for other ids)
 *   token i is accepted when u_accept[b,i] < p_i(x_i) / q_i(x_i) (always when q_i(x_i) = 0)
 *   n_accept[b] = n, the number of leading accepted tokens
 *   token[b]    = the emitted token: n < L: a draw from max(0, p_n - q_n); n = L: a draw from p_L;
 *                 drawn by inverse CDF in vocabulary order: the smallest v whose running sum of the
 *                 weights exceeds u_sample[b] times their total (a zero total: the weights p_n)
 * The uniforms are inputs, so a call is deterministic; decisions are taken in fp32, so where a
 * uniform lies within rounding of its threshold the outcome may differ from exact arithmetic.
 *
 * logits [B x (L+1) x vocab]: device, `dtype` (finite values), 16-byte aligned rows.
 * cand_idx int32, cand_prob fp32 [B x L x K]; draft_token int32, u_accept fp32 [B x L]; u_sample
 * fp32 [B] (uniforms in [0, 1)): device; the L-sized inputs may be NULL when L = 0.
 * n_accept_out, token_out int32 [B]: device.  0 <= L <= 64, K <= DH_MAX_K (K >= 1 when L > 0),
 * temperature > 0 and finite.  Workspace: dh_verify_chain_workspace bytes (256-byte aligned; need
 * not be zeroed).  B = 0 is a no-op.
 * ------------------------------------------------------------------------------------------- */
size_t dh_verify_chain_workspace(int B, int L, int vocab, int dtype);
int dh_verify_chain(const void* logits, const int32_t* cand_idx, const float* cand_prob, const int32_t* draft_token,
                    const float* u_accept, const float* u_sample, int B, int L, int vocab, int K, int dtype,
                    float temperature, int32_t* n_accept_out, int32_t* token_out, void* workspace, size_t ws_bytes,
                    void* stream);

/* ---------------------------------------------------------------------------------------------
 * Greedy draft-tree acceptance without a caller-provided workspace (no counterpart on the pages:
 * it is an interface for callers, not part of the method).
 *
 * For callers that cannot allocate device memory, such as code inside a serving engine's step
 * where cudaMalloc is not allowed (it can synchronise the device), or a host program that only
 * receives device pointers.  Same inputs, outputs and results as dh_tree_accept; the per-node
 * scratch lives in a fixed array inside the library's device memory, so the call allocates
 * nothing.  Limit: B * N <= DH_TREE_NOALLOC_MAX_NODES (larger calls return DH_ERR_UNSUPPORTED and
 * dh_last_error says why).  Every call looks up the array's device address in the current context
 * (a host-side query, so the address stays right after a device reset); the first call on a device
 * may load the library's device code, so make it before any stream capture.  All calls on a device
 * share the array, so calls whose kernels overlap on the GPU race on it: order them (one stream).
 * ------------------------------------------------------------------------------------------- */
#define DH_TREE_NOALLOC_MAX_NODES (1 << 18)
int dh_tree_accept_noalloc(const void* logits, const int32_t* parent, const int32_t* token, int B, int N,
                           int vocab, int dtype, int32_t* argmax_out, int32_t* path_out, int32_t* len_out,
                           int32_t* bonus_out, int32_t* err_out, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Device-side status of a workspace (no counterpart on the pages).
 *
 * Kernels that wait on on-chip barriers give up after a bounded time instead of hanging; they then
 * set bit (1 << DH_ERR_TIMEOUT) in the first word of the workspace they ran with, and their outputs
 * for that call are unspecified.  dh_workspace_status copies that word to *status_out (0 = no
 * event), clears it, and synchronises `stream`.  workspace: device, 256-byte aligned.
 * ------------------------------------------------------------------------------------------- */
int dh_workspace_status(void* workspace, void* stream, int* status_out);

/* ---------------------------------------------------------------------------------------------
 * Self-test of the bounded device-side waits (no counterpart on the pages).
 *
 * Queues one small kernel that waits, with the code the pipelined kernels use for their TMA,
 * bulk-copy and MMA completions, on an mbarrier that nothing arrives at (mode must be 0).  The wait
 * gives up after limit_us microseconds (1..1000000) and raises bit (1 << DH_ERR_TIMEOUT) in the
 * workspace status word, which dh_workspace_status then reports; the CUDA context stays usable.
 * workspace: a zero-filled device buffer of at least 256 bytes, 256-byte aligned.
 * ------------------------------------------------------------------------------------------- */
int dh_selftest_wait_timeout(int mode, int limit_us, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Kernel timing for measurement (no counterpart on the pages).
 *
 * dh_prof_enable(1) makes every subsequent call record a CUDA event pair around each kernel it
 * launches, on the caller's stream (this serialises the calls' kernels; do not enable it while a
 * stream is being captured).  dh_prof_enable(0) stops recording.  dh_prof_read waits for the
 * recorded events, and for up to max_kernels distinct kernels fills names (NUL-terminated, at most
 * name_len bytes each, packed at stride name_len), total_ms and launches; it returns the number of
 * distinct kernels (or -1 on a CUDA error) and clears the record.
 * ------------------------------------------------------------------------------------------- */
int dh_prof_enable(int on);
int dh_prof_read(char* names, int name_len, double* total_ms, int* launches, int max_kernels);

/* ---------------------------------------------------------------------------------------------
 * Test and tuning switches (no counterpart on the pages): which kernels serve a call.  Results do
 * not depend on them beyond the choice of kernels.
 *
 * Each switch is read once per process from the environment variable of the same name, on the
 * library's first use of it, and afterwards changes only through this call.  name / value:
 *   "DH_FORCE_PATH"    "auto" | "gemv" | "mma" | "fused"  stage-1 path, when it supports the shape
 *   "DH_FORCE_HEAD"    "auto" | "split" | "cluster"      dh_draft_head without the cluster head, or
 *                                                        with it wherever it fits, whatever K
 *   "DH_HEAD_CTAS"     "16" | "8" | "4" | "2"            largest cluster of the fused head
 *   "DH_FORCE_RESCORE" "auto" | "direct" | "ring" | "ticket" | "sweep" | "bucket"  stage-2 kernel
 *                      ("bucket": the ring kernel in its vocabulary-bucket mode at any size)
 *   "DH_SCORES_SMALL"  "lsu" | "tma"                     small-batch scores kernel
 *   "DH_HEAD_SELECT"   "auto" | "radix"                  fused head: the cooperative radix selection
 *                                                        instead of the group-best threshold
 * value NULL or "" restores the default.  Unknown names or values return DH_ERR_INVALID_ARG.  Not
 * synchronised with calls running on other host threads: set switches before such calls.
 * ------------------------------------------------------------------------------------------- */
int dh_set_tuning(const char* name, const char* value);

#ifdef __cplusplus
}
#endif

#endif /* DH_H */
