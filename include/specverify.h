/*
 * libspecverify: the verify-and-commit step of speculative decoding, on one GPU.
 *
 * Given the target model's logits for an anchor plus its draft positions, each
 * call scans every vocabulary row once on the GPU, decides how many drafts are
 * accepted, produces the correction / bonus token, and emits the KV-commit
 * index lists for the accepted positions.  Each round yields r + 1 tokens
 * (r accepted drafts plus one correction or bonus).
 *
 * Sources, cited as page title and section:
 *   [E2D] "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理"
 *         (tom-jerr.github.io/sglang/eagle2-in-sglang)
 *   [SGO] SGLang speculative-decoding overview (zdszero.github.io/speculative_decoding.html)
 *
 * Row convention (row-aligned verify input, [E2D] §1.1 and the verify_ids_2d
 * construction in §5.6): the target runs on [a, d1 .. dm]; row i of a request
 * carries input token verify_ids[i] (the anchor a at the request's first row)
 * and its logits give the distribution that tests verify_ids[i + 1].  The last
 * row of a request is only used for the bonus token.
 *
 * Memory and execution rules shared by every entry point:
 *   - Every array argument is a DEVICE pointer owned by the caller.  The
 *     library never allocates, never synchronises the stream and never reads
 *     device memory from the host; all work is enqueued on `stream`.
 *   - logits: [rows, ld] row-major, fp32 or bf16 (raw bits), ld >= vocab.  The
 *     base pointer must be 16-byte aligned and ld * element_size a multiple of
 *     16.  The same rules hold for q ([rows, ldq] fp32).
 *   - Host-side argument errors return a status code before anything is
 *     enqueued.  Data errors found on the device are reported per request in
 *     out->dev_status (bits below) and still produce defined outputs.
 *   - ws / ws_bytes: scratch of at least spec_verify_workspace_bytes(...)
 *     bytes, 256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE.  Every call
 *     whose kernels run to completion leaves the workspace's counter words at
 *     zero again, so a workspace can be reused by later calls on the same
 *     stream without clearing.  Calls that share a workspace must not overlap
 *     on the GPU.
 *   - Temperature: a request with temperature T samples iff 1e-30 <= T < inf;
 *     any other value (0, negative, NaN, inf) verifies that request greedily
 *     ([E2D] §6.5: greedy rows carry a one-hot q).
 *   - Uniforms are supplied by the caller in [0, 1): u_accept[row] decides the
 *     acceptance test at that row (for trees: at that node's row), u_final[b]
 *     draws the request's one correction / bonus token.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_NULL_ARG = 1,            /* a required pointer is NULL                        */
  SV_ERR_BAD_SHAPE = 2,           /* a size, stride or scalar argument is out of range */
  SV_ERR_BAD_DTYPE = 3,           /* dtype is not SV_F32 or SV_BF16                    */
  SV_ERR_MISALIGNED = 4,          /* a base pointer or row stride breaks 16-byte rule  */
  SV_ERR_UNSUPPORTED = 5,         /* a combination the library does not implement     */
  SV_ERR_WORKSPACE_TOO_SMALL = 6, /* ws is NULL, too small or not 256-byte aligned     */
  SV_ERR_CUDA = 7                 /* a CUDA launch or device query failed              */
} sv_status_t;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype_t;

/* Per-request device status bits (out->dev_status[b], OR-ed). */
#define SV_DEV_TOKEN_RANGE 1u    /* a tested draft / child token is outside [0, vocab): it is rejected   */
#define SV_DEV_NONFINITE 2u      /* a visited row had NaN / +inf entries (ignored) or was all -inf;      */
                                 /* an all -inf row stops verification there and its token is -1          */
#define SV_DEV_BAD_TREE 4u       /* parents / sibling lists invalid: the request is verified as its root  */
#define SV_DEV_BAD_LAYOUT 8u     /* cu_seqlens range invalid: nothing committed, num_out 0, bonus -1      */
#define SV_DEV_RESIDUAL_EMPTY 16u /* residual mass was <= 0: the token was sampled from p instead         */
#define SV_DEV_DUP_SIBLING 32u   /* target-only tree: a sibling repeats a token; the repeat is skipped    */
#define SV_DEV_TIMEOUT 64u       /* a bounded wait inside a kernel gave up (never expected): this call's   */
                                 /* outputs are undefined and the workspace must be zero-filled again      */

/*
 * Outputs of one call (all DEVICE pointers, caller-owned).  max_len is the
 * per-request row bound of the call (chains: m + 1; ragged: max_len; trees:
 * nodes).  [E2D] §5.6.6 and §8.1 table; [SGO] "两个容易误解的工程细节".
 */
typedef struct {
  int32_t* accept_len;      /* [B] r, accepted drafts                                        */
  int32_t* num_out;         /* [B] r + 1 (= commit_lens); 0 for a bad layout                  */
  int32_t* out_tokens;      /* [B, max_len] accepted drafts then the bonus; rest -1           */
  int32_t* bonus;           /* [B] correction / bonus token (-1 when no usable row)          */
  int32_t* accept_rows;     /* [B, max_len] global logits rows committed: anchor row, then    */
                            /*   the rows of the accepted drafts / tree path; rest -1          */
  int32_t* commit_cu;       /* [B + 1] exclusive scan of num_out                              */
  int64_t* commit_src_slot; /* [rows] or NULL: row_slots[accept_rows[b][k]] at commit_cu[b]+k */
  int64_t* commit_dst_pos;  /* [rows] or NULL: seq_lens[b] + k at commit_cu[b] + k            */
  uint32_t* dev_status;     /* [B] SV_DEV_* bits                                              */
} sv_out_t;

/* Bytes of workspace needed for a call with these sizes (rows = total logits
 * rows, max_len = per-request row bound / tree nodes). */
size_t spec_verify_workspace_bytes(int64_t rows, int32_t batch, int32_t vocab, int32_t max_len);

/* Static description of a status code. */
const char* spec_verify_status_string(sv_status_t status);

/* Description of the CUDA error behind the last SV_ERR_CUDA returned on this
 * host thread ("no error" if none). */
const char* spec_verify_last_cuda_error(void);

/* Benchmark instrumentation (not needed for verification).  While set, every
 * call made from this host thread records `start` on its stream immediately
 * before its row-statistics kernel and `stop` immediately after it, so the
 * caller can time that kernel with cudaEventElapsedTime.  The events are the
 * caller's; pass NULL, NULL to stop.  Returns SV_ERR_NULL_ARG if exactly one
 * of the two is NULL. */
sv_status_t spec_verify_set_stats_events(cudaEvent_t start, cudaEvent_t stop);

/*
 * Greedy chain verification ([E2D] §1.2 first bullet; [SGO] "为什么结果不受
 * draft 影响": accept while the target argmax equals the draft, else replace
 * it with the argmax and stop).  batch requests of m drafts each: rows =
 * batch * (m + 1), request b owns rows [b*(m+1), (b+1)*(m+1)).  Argmax ties
 * resolve to the lowest index.  row_slots [rows] and seq_lens [B] (int64) are
 * only needed for commit_src_slot / commit_dst_pos.
 */
sv_status_t spec_verify_greedy_chain(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m,
                                     int32_t vocab, const int32_t* verify_ids, const int64_t* row_slots,
                                     const int64_t* seq_lens, const sv_out_t* out, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

/*
 * Greedy tree verification ([SGO] "为什么结果不受 draft 影响", verify_tree_greedy;
 * [E2D] §2.4, §3.4).  Request b has `nodes` nodes (node 0 = root / anchor);
 * node i owns logits row b*nodes + i, carries token tokens[b][i] and has parent
 * parents[b][i] (-1 for the root, otherwise 0 <= parent < i).  From the root,
 * the walk moves to the first child (ascending node index, or the order of the
 * optional first_child / next_sibling lists, both [B, nodes], -1 terminated)
 * whose token equals the current row's argmax; the bonus is the argmax of the
 * last node's row.  nodes <= 1024.
 */
sv_status_t spec_verify_greedy_tree(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t nodes,
                                    int32_t vocab, const int32_t* tokens, const int32_t* parents,
                                    const int32_t* first_child, const int32_t* next_sibling,
                                    const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out,
                                    void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * p/q rejection chain ([E2D] §1.2: alpha = min(1, p/q), residual
 * p' = [p - q]_+ / sum [p - q]_+; temperature-scaled softmax p = softmax(l/T),
 * §6.2).  Row j of a request accepts its draft d iff u_accept[row] * q[row][d]
 * < p_row(d); at the first rejection the correction is drawn from the residual
 * of that row, and when every draft passes the bonus is drawn from p of the
 * last row.  Draws use inverse CDF: the smallest v whose running weight sum
 * exceeds u_final[b] * S (§6.2, sample_path()).  q [rows, ldq] fp32 is the
 * proposal actually sampled from ([E2D] §5.6.1, §6.5); the last row of each
 * request is never read.  temperature [B], u_accept [rows], u_final [B] fp32.
 */
sv_status_t spec_verify_rejection_chain(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch, int32_t m,
                                        int32_t vocab, const int32_t* verify_ids, const float* q, int64_t ldq,
                                        const float* temperature, const float* u_accept, const float* u_final,
                                        const int64_t* row_slots, const int64_t* seq_lens, const sv_out_t* out,
                                        void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Verification by independent target sampling and prefix match ([E2D] §1.2:
 * a verification of its own, distinct from p/q rejection; the DFlash
 * inference loop: sample the target's posterior at every block position, the
 * accept length is the longest prefix where draft and sample agree, and the
 * first mismatch emits the sample).  Same layout and outputs as
 * spec_verify_rejection_chain, without q: row i's target token is drawn by
 * inverse CDF with u_sample[i] (argmax for a greedy request), draft
 * verify_ids[i + 1] is accepted iff it equals that draw, and the first
 * rejected row (or the last row when every draft is accepted) emits its own
 * draw.  No row is drawn in full except the one emitting: the statistics pass
 * also sums each row's probabilities below its draft token, and the draw
 * equals the draft iff u * Z lies in [that sum, that sum + p(draft) * Z).
 * ws: spec_verify_workspace_bytes(batch * (m + 1), batch, vocab, m + 1) bytes.
 */
sv_status_t spec_verify_sample_match_chain(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                           int32_t m, int32_t vocab, const int32_t* verify_ids,
                                           const float* temperature, const float* u_sample, const int64_t* row_slots,
                                           const int64_t* seq_lens, const sv_out_t* out, void* ws, size_t ws_bytes,
                                           cudaStream_t stream);

/*
 * p/q rejection chain with a SPARSE q ([E2D] §6.2, §6.5: a candidate selector
 * proposes from K candidates; its q is zero outside them, and tokens outside
 * the candidates can still come out through the residual [p - q]_+).  Same
 * arguments and results as spec_verify_rejection_chain, with q replaced by
 * candidate lists: cand_ids / cand_probs [rows, ldc] (device int32 / fp32,
 * ldc >= num_cands, 1 <= num_cands <= 1024); row i's list describes the q that
 * proposed verify_ids[i + 1]: q_i(v) = the sum of cand_probs[i][c] over c with
 * cand_ids[i][c] == v.  Id -1 is padding; any other id outside [0, vocab) is
 * ignored and sets SV_DEV_TOKEN_RANGE for the request when it appears in one of
 * the request's tested rows (all rows but its last).  No dense q is read or
 * formed; the final draw of a rejected request reads that row's list in place,
 * so the lists, like every input, must stay unchanged until the call's work on
 * the stream has completed.  ws: at least
 * spec_verify_sparse_workspace_bytes(batch * (m + 1), batch, vocab, m + 1,
 * num_cands) bytes (same rules as every workspace; num_cands does not change
 * the size).
 */
size_t spec_verify_sparse_workspace_bytes(int64_t rows, int32_t batch, int32_t vocab, int32_t max_len,
                                          int32_t num_cands);

sv_status_t spec_verify_rejection_chain_sparse(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                               int32_t m, int32_t vocab, const int32_t* verify_ids,
                                               const int32_t* cand_ids, const float* cand_probs, int32_t num_cands,
                                               int64_t ldc, const float* temperature, const float* u_accept,
                                               const float* u_final, const int64_t* row_slots,
                                               const int64_t* seq_lens, const sv_out_t* out, void* ws,
                                               size_t ws_bytes, cudaStream_t stream);

/*
 * Ragged p/q rejection ([E2D] §5.6.5: verify_lens include the anchor, compact
 * offsets, e.g. lens [4,2,6] -> [0,4,6,12]).  Request b owns rows
 * [cu_seqlens[b], cu_seqlens[b+1]) of the total_rows rows; lengths must lie in
 * [1, max_len] (length 1 = bonus only).  A request whose range is invalid gets
 * SV_DEV_BAD_LAYOUT and commits nothing.  Otherwise as the rejection chain.
 */
sv_status_t spec_verify_rejection_ragged(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                         int64_t total_rows, int32_t max_len, int32_t vocab,
                                         const int32_t* cu_seqlens, const int32_t* verify_ids, const float* q,
                                         int64_t ldq, const float* temperature, const float* u_accept,
                                         const float* u_final, const int64_t* row_slots, const int64_t* seq_lens,
                                         const sv_out_t* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Target-only tree sampling ([SGO] "为什么结果不受 draft 影响":
 * tree_speculative_sampling_target_only uses only target probabilities, draft
 * probabilities passed as 0, thresholds default 1.0).  At node cur with
 * uniform u = u_accept[row(cur)], children are visited in order with
 * c += p_cur(token); the first child with u < c / threshold_acc or
 * p_cur(token) >= threshold_single is accepted.  A sibling repeating an
 * earlier sibling's token is skipped (SV_DEV_DUP_SIBLING).  If no child is
 * accepted the final token is drawn from p_cur with the children's tokens
 * zeroed; at a leaf, from p_leaf.  With both thresholds 1.0 the output law
 * equals the target's.  threshold_acc must be > 0 and finite.  Tree layout as
 * in spec_verify_greedy_tree.
 */
sv_status_t spec_verify_target_only_tree(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                         int32_t nodes, int32_t vocab, const int32_t* tokens,
                                         const int32_t* parents, const int32_t* first_child,
                                         const int32_t* next_sibling, const float* temperature,
                                         float threshold_single, float threshold_acc, const float* u_accept,
                                         const float* u_final, const int64_t* row_slots, const int64_t* seq_lens,
                                         const sv_out_t* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * p/q rejection chain without a caller workspace.  (The pages have no
 * counterpart: this is a deployment convenience of this library.)
 *
 * For callers that cannot provide device scratch memory — for example a plugin
 * that its host framework hands only input and output buffers, code that runs
 * after a serving engine has reserved all device memory for itself, or an
 * embedding that must not allocate at call time.  Same arguments and results as
 * spec_verify_rejection_chain, minus ws / ws_bytes: the library uses one fixed
 * scratch area of SV_NOALLOC_SCRATCH_BYTES bytes in its own device image (every
 * GPU that uses the library keeps it until the process exits) and allocates
 * nothing.  Problems whose workspace would exceed that size
 * (spec_verify_workspace_bytes(batch*(m+1), batch, vocab, m+1) >
 * SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE_TOO_SMALL, and argument
 * errors their status code, before anything is enqueued or any CUDA call is
 * made.  The first call in each CUDA context (on each device, and again after a
 * device reset) looks up the area's device address; make it before any stream
 * capture starts.  Every call clears the area's counter words on `stream` before
 * launching; all calls share the area, so calls that overlap on the GPU (other
 * streams or host threads) race — serialise them.
 */
#define SV_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

sv_status_t spec_verify_rejection_chain_noalloc(const void* logits, sv_dtype_t dtype, int64_t ld, int32_t batch,
                                                int32_t m, int32_t vocab, const int32_t* verify_ids, const float* q,
                                                int64_t ldq, const float* temperature, const float* u_accept,
                                                const float* u_final, const int64_t* row_slots,
                                                const int64_t* seq_lens, const sv_out_t* out, cudaStream_t stream);

/*
 * Test and diagnostic hooks (the pages have no counterpart; not for production use).
 *
 * spec_verify_noalloc_fill_counters sets every byte of the no-allocation scratch
 * area's counter words (the words each spec_verify_rejection_chain_noalloc call
 * clears before it launches) to value & 0xff, on `stream`, in the current
 * context: a test uses it to show that a call does not depend on what an earlier
 * call left there.  Returns SV_ERR_CUDA if the area cannot be reached.
 *
 * spec_verify_set_hand_off_limit_ns(ns), ns > 0, puts the row-statistics kernel
 * of every later call, in every thread, into its expiry test: each in-CTA
 * hand-off wait gives up after ns nanoseconds, and one wait on a barrier that
 * nothing completes is sure to; the kernel then stops, waits (with the normal
 * one-second limit) for its own bulk copies still in flight, and raises the
 * workspace error word, so the call's requests report SV_DEV_TIMEOUT.  ns = 0
 * (the default) restores normal operation.  After a timed-out call, zero-fill
 * the workspace before using it again.  Always returns SV_OK.
 */
sv_status_t spec_verify_noalloc_fill_counters(uint32_t value, cudaStream_t stream);
sv_status_t spec_verify_set_hand_off_limit_ns(uint64_t ns);

/*
 * Row statistics on their own (the single pass every entry point starts
 * with; [E2D] §1.2 and §6.2: the target distribution of a row is
 * softmax(l / T), and a greedy row takes its argmax): for each of `rows`
 * rows, the maximum M (float), the lowest argmax (-1 for an all -inf row),
 * Z = sum_v exp((l_v - M)/T) with T = row_temp[row] (0 when row_temp is NULL
 * or the row is greedy), p at probe[row] (when probe and out_p are given),
 * and SV_DEV_NONFINITE in row_flags.  out_z is double.  All outputs [rows],
 * device, caller-owned; out_p / probe / row_temp may be NULL.  ws: at least
 * spec_verify_workspace_bytes(rows, 1, vocab, 1) bytes (same rules as every
 * workspace).  Argument errors (SV_ERR_NULL_ARG for a missing logits,
 * out_max, out_argmax or out_z; the logits checks of every entry point)
 * return before anything is enqueued.
 */
sv_status_t spec_verify_row_stats(const void* logits, sv_dtype_t dtype, int64_t ld, int64_t rows, int32_t vocab,
                                  const float* row_temp, const int32_t* probe, float* out_max,
                                  int32_t* out_argmax, double* out_z, float* out_p, uint32_t* row_flags,
                                  void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * DSpark verify-length scheduling ([E2D] §5.6.3 host budget, §5.6.4 device
 * allocation): how many draft rows each request verifies in the next round.
 *
 * spec_verify_dspark_budget runs on the HOST (no GPU, host pointers).  It picks
 * the extra draft budget K from historical survival scores: hist_survival[n]
 * holds one score per (request, draft position) in any order; NaN scores and
 * scores below eps are dropped, the rest sorted descending a_1 >= a_2 >= ...;
 * with N(K) = R + a_1 + ... + a_K (predicted committed tokens) and sps[M] the
 * speed (rounds per second) of a round with M target rows, M = 0 .. sps_len-1,
 *   *k_star = argmax over K with R + K < sps_len of N(K) * sps[R + K]
 * (the smaller K on ties; 0 when R >= sps_len).  Returns SV_ERR_NULL_ARG or
 * SV_ERR_BAD_SHAPE (n < 0, num_requests < 0, sps_len < 0) on bad arguments.
 *
 * spec_verify_dspark_verify_lens runs on the DEVICE.  survival [R, D] (device
 * fp32, row stride ld >= D floats) holds each request's current survival at
 * draft positions 1..D (a running product of confidences, so non-increasing
 * along a row).  Every (request r, position j) is a candidate; candidates are
 * ordered by survival descending, then position ascending, then request
 * ascending (no token id enters the order), and the first `budget` whose
 * survival is at least eps are selected (NaN orders last and is never
 * selected).  verify_lens[r] = clamp(1 + selected_r, min_len, max_len): one
 * anchor row plus the selected drafts (device int32 [R]).  ws: at least
 * spec_verify_dspark_workspace_bytes(R) bytes, zero-filled before its first
 * use; each completed call leaves it zeroed.  Host argument errors
 * (SV_ERR_NULL_ARG, SV_ERR_BAD_SHAPE for R, D or budget < 0, ld < D,
 * min_len < 1, max_len < min_len, R * D > 2^30; SV_ERR_WORKSPACE_TOO_SMALL)
 * return before anything is enqueued.
 */
size_t spec_verify_dspark_workspace_bytes(int32_t num_requests);

sv_status_t spec_verify_dspark_budget(const float* hist_survival, int64_t n, int32_t num_requests, const float* sps,
                                      int32_t sps_len, float eps, int32_t* k_star);

sv_status_t spec_verify_dspark_verify_lens(const float* survival, int32_t num_requests, int32_t num_drafts,
                                           int64_t ld, int32_t budget, int32_t min_len, int32_t max_len, float eps,
                                           int32_t* verify_lens, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Tree-verify inputs from parent lists ([E2D] §2.4: a flattened tree where each
 * node sees the committed history, its ancestors and itself, with position ids
 * from the path depth; §3.4: tree construction produces the mask, positions
 * and the retrieve index / next-token / next-sibling arrays of the verify walk).
 * parents [batch, nodes] (device int32): node 0 is the root (parent -1), every
 * other node's parent has a smaller index.  seq_lens [batch] (device int64,
 * may be NULL for 0): the committed length before the tree.  Outputs, all
 * device, caller-owned:
 *   positions      [batch, nodes] int64  seq_len + depth
 *   mask           [batch, nodes, nodes] uint8, mask[b][i][j] = 1 iff node j
 *                  is node i or one of its ancestors
 *   retrieve_index [batch, nodes] int32  b * nodes + i
 *   first_child    [batch, nodes] int32  lowest-index child, -1 if none
 *   next_sibling   [batch, nodes] int32  next higher-index node with the same
 *                  parent, -1 if none (the format the tree entry points accept)
 *   status         [batch] uint32        SV_DEV_BAD_TREE for an invalid parent
 *                  array (its outputs: depth 0, identity mask, -1 links)
 * 1 <= nodes <= 1024, batch <= 65535; SV_ERR_BAD_SHAPE / SV_ERR_NULL_ARG
 * before anything is enqueued.  No workspace.
 */
sv_status_t spec_verify_build_tree(const int32_t* parents, const int64_t* seq_lens, int32_t batch, int32_t nodes,
                                   int64_t* positions, uint8_t* mask, int32_t* retrieve_index,
                                   int32_t* first_child, int32_t* next_sibling, uint32_t* status,
                                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
