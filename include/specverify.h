/*
 * specverify.h - C ABI of the GB300 speculative-decoding verification library.
 *
 * The library implements the verifier-side step of speculative decoding:
 *   - spec_verify_sample: temperature softmax of target and draft logits,
 *     the accept/reject test of each draft token, the first rejection, and the
 *     correction (residual) or bonus draw;
 *   - spec_verify_greedy: the argmax-match variant;
 *   - spec_verify_tree_greedy: greedy verification of a draft tree;
 *   - kv_commit_rollback: commit of the accepted provisional KV slots into a
 *     paged cache and release of the provisional blocks.
 *
 * Sources (page title, section):
 *   [L] aiengineeringfromscratch.com, "Speculative decoding and EAGLE-3":
 *       "Variant: Leviathan rejection sampling" (accept d ~ p with probability
 *       min(1, q(d)/p(d)); on rejection sample (q - p)+ / ||(q - p)+||_1; the
 *       verifier returns q_1..q_{N+1}; first rejection at j samples the
 *       residual of row j, full acceptance samples a bonus token from
 *       q_{N+1}); "Step 1: the rejection rule" (p(d) <= 0 accepts; strict
 *       u < min(1, q/p)); "Step 2: residual distribution" (zero residual mass
 *       falls back to q); "Rolling back the KV cache" and "Step 4: KV rollback
 *       accounting" (logical length prefix + j + 1).
 *   [P] devpost.com, "phoenix", section "What it does": greedy verification
 *       keeps tokens up to the first disagreement and writes the target's token
 *       there; output identical to the target alone.
 *   [S] "sglang_spec_decode" README, provisional KV layer: provisional blocks
 *       are committed or freed immediately; no block leaked or freed twice.
 *   [Q] quickscale.ai, "Quand et pourquoi utiliser le speculative decoding":
 *       "Influence du sampling" (temperature, top-p, top-k shape the verified
 *       distributions); per-position acceptance, mean acceptance length.
 *   [G] thakicloud.com, "Speculative decoding: when it loses", section "Grading
 *       every branch in one pass": draft branches flattened under an ancestor-only
 *       mask, graded in one target pass, the longest surviving path kept; [L]
 *       "EAGLE-2" (dynamic draft tree) and its [2, 2, 2] tree exercise.
 *
 * Notation: q = target (verifier) distribution, p = draft distribution.
 * Positions are 0-based: draft positions 0..K-1, bonus row K.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller. The library
 *     allocates no device or host memory and keeps no state between calls
 *     (its only static data is a read-only constant table, a per-process cache
 *     of occupancy queries and, as the one exception, the 4 MiB writable
 *     device scratch of spec_verify_greedy_noalloc, which all of that entry
 *     point's calls on a device share). The verify calls take a caller-allocated
 *     device workspace of spec_verify_workspace_bytes(B, K, V, dtype) bytes
 *     (256-byte aligned) that holds per-slice partial sums and the work queue;
 *     its contents need no initialisation, and calls that share one workspace
 *     must not overlap on the device (one stream, or ordered streams).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream). Nothing synchronises; outputs are valid once
 *     the stream reaches the call.
 *   - Arguments are validated on the host before any launch. A host-side
 *     failure returns a negative status and launches nothing.
 *   - Problems only visible on the device (a token id out of range, non-finite
 *     logits, an exhausted free-block stack) are reported by OR-ing bits into
 *     the optional device word *err_flag; the affected batch row is written
 *     as -1 (verify) or the whole call leaves its state unchanged (KV commit).
 *     No device-side trap or assert is ever raised.
 *   - Arrays are C-contiguous. Logit arrays must start on a 16-byte boundary.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ---- */
#define SPEC_OK 0
#define SPEC_EINVAL (-1)   /* null pointer, bad size, bad dtype, misaligned logits */
#define SPEC_ECUDA (-2)    /* a CUDA launch or attribute call failed */
#define SPEC_ENOTSUP (-3)  /* valid request this build does not handle */

/* ---- logit dtypes ---- */
#define SPEC_BF16 0 /* bfloat16, passed as raw 16-bit words */
#define SPEC_F32 1  /* IEEE float32 */

/* ---- device error bits OR-ed into *err_flag ---- */
#define SPEC_DERR_TOKEN 1        /* a draft token outside [0, V); that row's outputs are -1 */
#define SPEC_DERR_LOGITS 2       /* a row needed by the step has NaN/+inf logits, only -inf, or
                                    (sampling, top-p) a maximum logit m with
                                    |m log2(e) / T| >= 2^18, beyond the exponent range */
#define SPEC_DERR_BAD_ACCEPT 4   /* kv: num_accepted outside [0, K] */
#define SPEC_DERR_BAD_LENGTH 8   /* kv: negative seq_len, or the row outgrows max_blocks */
#define SPEC_DERR_NO_SPACE 16    /* kv: the free stack cannot supply every new block */
#define SPEC_DERR_BAD_BLOCK 32   /* kv: a block id out of range, or a target slot already taken */
#define SPEC_DERR_TIMEOUT 64     /* an internal bounded wait gave up (should never happen);
                                    the launch drains and unfinished rows' outputs are not
                                    written. Failure-detection tests provoke it with the
                                    environment knobs SPECVERIFY_STALL_ROW=b (every stage
                                    arrival of batch row b is withheld) and
                                    SPECVERIFY_IDLE_NS (the producers' idle limit, default
                                    2 s), read at every verify launch */
#define SPEC_DERR_BAD_SLOT 128   /* kv: a slot_map entry of a kept position outside [0, K] */

/* ---- per-row diagnostic bits written to row_info[b] (optional) ---- */
#define SPEC_ROW_ACCEPT_REFINED 1 /* an accept test fell inside the fp32 error bound and was
                                     decided by the double-float path */
#define SPEC_ROW_SAMPLE_REFINED 2 /* the final draw fell inside the error bound of its first
                                     pass (the fp32 sweep; for batches of 4 to 48 rows, a
                                     residual draw's first pass is the accurate lite pass)
                                     and was decided by a more accurate one */
#define SPEC_ROW_UNCERTIFIED 4    /* the double-float path could not certify its decision either
                                     (its result is still returned) */
#define SPEC_ROW_ZERO_RESIDUAL 8  /* the residual mass was exactly zero; q_j was used */

/*
 * spec_verify_sample - accept/reject with temperature softmax ([L] Leviathan
 * rejection sampling, Steps 1-3).
 *
 *   target_logits  [B, K+1, V]  dtype  target row i is q_i before softmax; row K is q_{K+1}
 *   draft_logits   [B, K,   V]  dtype  draft row i is p_i before softmax
 *   draft_tokens   [B, K]       int32  d_i, expected in [0, V)
 *   uniforms       [B, K+1]     float  in [0, 1): u[i] decides test i, u[K] is the single
 *                                      uniform of the correction or bonus draw
 *   temperature    > 0 applies softmax(z / T) to both tensors; == 0 behaves exactly as
 *                  spec_verify_greedy (draft_logits and uniforms are then unused);
 *                  negative or NaN -> SPEC_EINVAL
 *   B >= 1, 1 <= K <= 31, V >= 1
 *   out_tokens       [B, K+1] int32  d_0..d_{n-1}, then the correction or bonus token, then -1
 *   out_num_accepted [B]      int32  n in [0, K] (-1 for a row with a device error)
 *   stream         cudaStream_t
 *   dtype          SPEC_BF16 or SPEC_F32 (both logit tensors)
 *   err_flag       optional [1] int32, device error bits are OR-ed in (never cleared)
 *   row_info       optional [B] int32, SPEC_ROW_* bits of each row (overwritten)
 *   q_at_d, p_at_d optional [B, K] float, q_i(d_i) and p_i(d_i) (for inspection)
 *   accept_counters optional [2K + 2] uint64, acceptance statistics ACCUMULATED over
 *                  calls (the caller zeroes it): [i] += rows in which draft position
 *                  i was tested (i <= n, i < K), [K + i] += rows in which it was
 *                  accepted (i < n), [2K] += rows verified, [2K + 1] += tokens
 *                  emitted (n + 1 per row). Rows with a device error are not
 *                  counted. Per-position acceptance a_i = [K+i] / [i]; mean
 *                  acceptance length = [2K+1] / [2K] ([Q] "mean acceptance length";
 *                  [L] expected accepted tokens).
 *   target_threshold optional [B, K+1] float, draft_threshold optional [B, K] float:
 *                  per-row logit thresholds from spec_filter_thresholds (top-k /
 *                  top-p); every token of a row whose logit is below the row's
 *                  threshold counts as logit -inf (probability 0) in the softmax,
 *                  the accept tests and the draw. Null: no filtering of that tensor.
 *                  Ignored in greedy mode (the argmax is never filtered).
 *
 * Semantics: for i = 0..K-1, d_i is accepted iff p_i(d_i) <= 0 or
 * u[i] < min(1, q_i(d_i)/p_i(d_i)); at the first rejection j the token is the
 * smallest v with u[K] * sum(r) < sum_{w<=v} r_w for r = max(0, q_j - p_j) (r = q_j if
 * that sum is 0); if all K are accepted the same draw is made from q_K. Every
 * decision is certified against a proven error bound of the arithmetic that took
 * it: the fp32 first pass, then for the decisions inside its bound a pass in pair
 * (double-float) arithmetic with a lighter exponential (relative error < 1e-9),
 * then, for what that leaves undecided, the full double-float pass (< 4e-13).
 * Batches of 4 to 48 rows start residual draws at the pair-arithmetic pass.
 * Logit arrays must be 16-byte aligned and V * sizeof(dtype) a multiple of 16.
 * workspace / workspace_bytes: see the conventions above (SPEC_EINVAL if too small).
 */
int spec_verify_sample(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* uniforms, float temperature,
                       int B, int K, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                       void* stream, int dtype, int32_t* err_flag, int32_t* row_info,
                       float* q_at_d, float* p_at_d, void* workspace, size_t workspace_bytes,
                       uint64_t* accept_counters, const float* target_threshold,
                       const float* draft_threshold);

/*
 * spec_verify_greedy - greedy verification ([P] "What it does").
 *
 *   target_logits [B, K+1, V] dtype; draft_tokens [B, K] int32.
 *   g_i = argmax_v target[b, i, v] over raw logits, ties to the lowest index.
 *   n = number of leading i with d_i == g_i; out_tokens[b] = d_0..d_{n-1}, g_n, -1...;
 *   out_num_accepted[b] = n. Same pointer, alignment and error conventions as
 *   spec_verify_sample; a row with NaN logits is reported as SPEC_DERR_LOGITS.
 *   accept_counters: optional, as for spec_verify_sample.
 */
int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int K,
                       int V, int32_t* out_tokens, int32_t* out_num_accepted, void* stream,
                       int dtype, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                       uint64_t* accept_counters);

/*
 * spec_verify_tree_greedy - greedy verification of a draft tree ([G]; [P] for
 * the greedy acceptance of one token).
 *
 *   target_logits [B, N+1, V] dtype: row 0 is the target after the committed
 *                 prefix, row 1 + i the target after draft node i (the target
 *                 ran once over the flattened tree with an ancestor-only mask).
 *   tree_parents  [B, N] int32: parent of node i, in [-1, i) (-1: a child of
 *                 the last committed token); nodes are in topological order.
 *   tree_tokens   [B, N] int32 in [0, V): the token of each node.
 *   1 <= N <= 31.
 *   g_r = argmax of row r (raw logits, ties to the lowest index). Node i is
 *   consistent when tree_tokens[i] == g of its parent's row (row parent + 1);
 *   it survives when it and all its ancestors are consistent. The kept path
 *   ends at the deepest survivor (the lowest node index among equally deep
 *   ones; none: empty path). With n = the path's length:
 *   out_tokens       [B, N+1] int32: the path's tokens, then g of its last
 *                    node's row (g_0 for an empty path), then -1;
 *   out_num_accepted [B] int32: n;
 *   out_slots        optional [B, N+1] int32: provisional KV slot of each kept
 *                    position, 0 (the last committed token) then 1 + node for
 *                    the path's nodes, then -1 (the slot_map of
 *                    kv_commit_rollback with K = N).
 *   With distinct sibling tokens the output equals target-only greedy decoding.
 *   An invalid parent or token sets SPEC_DERR_TOKEN; a NaN in row 0 or in the
 *   row of a surviving node sets SPEC_DERR_LOGITS; such a row's outputs are -1.
 *   Workspace: spec_verify_workspace_bytes(B, N, V, dtype). Other conventions
 *   as spec_verify_greedy.
 */
int spec_verify_tree_greedy(const void* target_logits, const int32_t* tree_parents,
                            const int32_t* tree_tokens, int B, int N, int V, int32_t* out_tokens,
                            int32_t* out_num_accepted, int32_t* out_slots, void* stream,
                            int dtype, int32_t* err_flag, void* workspace,
                            size_t workspace_bytes);

/*
 * spec_filter_thresholds - top-k / top-p logit threshold of every row
 * ([Q] "Influence du sampling" names temperature, top-k and top-p as the
 * parameters shaping the verified distributions; the pages define neither).
 *
 *   logits        [R, V] dtype (SPEC_BF16 or SPEC_F32), 16-byte aligned rows
 *                 (V * sizeof(dtype) a multiple of 16)
 *   temperature   > 0 (top-p is taken on softmax(z / T); top-k ignores T)
 *   top_k         0 (off) or k: keep the tokens whose logit is >= the k-th
 *                 largest logit of the row (ties all kept; k >= V is off)
 *   top_p         in (0, 1] (1 is off): on the renormalised top-k distribution,
 *                 keep the tokens whose logit is >= t*, the largest logit value
 *                 t at which the tokens with logit >= t reach probability p
 *                 (ties all kept)
 *   out_threshold [R] float: the row's threshold (keep z >= threshold); -inf when
 *                 nothing is filtered; +inf for a row with a NaN logit, or with
 *                 top-p a maximum logit out of range (see SPEC_DERR_LOGITS; its
 *                 verification then reports SPEC_DERR_LOGITS; the bit is also set here)
 *   err_flag      optional [1] int32, device error bits OR-ed in
 * Top-k is an exact integer selection. Top-p compares exactly summed fixed-point
 * masses whose per-token error is bounded; a row whose comparison falls inside
 * the fp32 bound is recomputed with double-float exponentials (error < 1e-11).
 * The thresholds feed spec_verify_sample's target_threshold / draft_threshold
 * (the same k and p for both tensors). Two kernels are enqueued on `stream`.
 */
int spec_filter_thresholds(const void* logits, int R, int V, int dtype, float temperature,
                           int top_k, float top_p, float* out_threshold, void* stream,
                           int32_t* err_flag);

/*
 * spec_verify_greedy_noalloc - spec_verify_greedy without a caller workspace.
 * The pages have no counterpart: this is a deployment variant for callers
 * that cannot hand the library a device allocation of their own, e.g. code
 * whose device memory is owned by another framework's pool, or plain C
 * callers with no device allocator at hand. The call itself allocates
 * nothing either: it uses one built-in device array of
 * spec_verify_greedy_noalloc_max_bytes() bytes (4 MiB), which every GPU that
 * loads the library holds until the process exits. Each call looks up the
 * array's address on the current device with cudaGetSymbolAddress; the first
 * call on a device may load the library's module there, so issue it before
 * any stream capture.
 *
 *   Arguments, outputs and errors: as spec_verify_greedy, without workspace.
 *   Returns SPEC_ENOTSUP when the step needs more scratch than the built-in
 *   array holds (spec_verify_workspace_bytes(B, K, V, dtype) > 4 MiB; e.g.
 *   B = 256, K = 4, V = 151936 bf16 needs about 3.0 MiB; B = 1024 steps with
 *   V >= 128256 need 9.8 to 12.4 MiB and are refused), SPEC_ECUDA when the
 *   array's address cannot be obtained.
 *   The scratch's counters and queue are cleared on `stream` at every call.
 *   All calls on one device share the array: calls that can overlap on the
 *   device race on it and must be ordered (one stream, or ordered streams).
 */
int spec_verify_greedy_noalloc(const void* target_logits, const int32_t* draft_tokens, int B,
                               int K, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                               void* stream, int dtype, int32_t* err_flag);

/* spec_verify_greedy_noalloc_max_bytes - size of the built-in scratch (bytes). */
size_t spec_verify_greedy_noalloc_max_bytes(void);

/*
 * spec_verify_workspace_bytes - size of the device workspace that
 * spec_verify_sample and spec_verify_greedy need for (B, K, V, dtype), and
 * spec_verify_tree_greedy for K = N; 0 for arguments those calls would reject.
 * One workspace serves all three calls. The size follows the work split, which
 * depends on B (batches of at most 48 rows for sampling, 64 for greedy, split
 * each row finer) and on the
 * test knob SPECVERIFY_SMALL_BATCH=0 or 1 (read from the environment here and
 * at every verify launch; it forces the small-batch split, per-position
 * first-stage tasks and residual draws starting at the refinement pass off or
 * on whatever B is, so that tests run both dispatches; the results are the
 * same either way). Query the size under the same setting as the launch.
 */
size_t spec_verify_workspace_bytes(int B, int K, int V, int dtype);

/*
 * kv_commit_rollback - commit the accepted provisional KV slots and free the
 * provisional blocks ([L] "Rolling back the KV cache", "Step 4"; [S] provisional layer).
 *
 *   block_table  [B, max_blocks] int32  committed blocks of each row, -1 = unused;
 *                                       entries [0, ceil(seq_len/bs)) must be valid
 *   seq_lens     [B] int32              committed length L_b; becomes L_b + n_b + 1
 *   num_accepted [B] int32              n_b from the verify call (same stream -> ordered)
 *   prov_blocks  [B, P] int32           blocks holding provisional slots 0..K
 *                                       (slot s in block prov[b][s / bs], offset s % bs);
 *                                       all are pushed to the free stack and set to -1
 *   kv_pool      [num_blocks][num_layers][2][block_size][num_kv_heads][head_dim]
 *                elements of kv_elem_bytes bytes (K and V planes per layer)
 *   free_stack   [num_blocks] int32, free_top [1] int32: a stack of free block ids,
 *                live entries free_stack[0 .. *free_top)
 *   status       REQUIRED [1] int32, overwritten on the device with 0 when the call
 *                committed, else with the SPEC_DERR_* bits that stopped it
 *   slot_map     optional [B, K+1] int32: kept position s takes the provisional
 *                slot slot_map[b][s] (entries s <= n must lie in [0, K], else
 *                SPEC_DERR_BAD_SLOT); null means slot s (the linear draft). A tree
 *                draft ([G]) passes the out_slots of spec_verify_tree_greedy.
 *   K            0 <= K <= 31; P (provisional blocks per row) in [1, 512];
 *                num_kv_heads * head_dim * kv_elem_bytes a multiple of 16, kv_pool
 *                16-byte aligned
 *
 * For every row, provisional slots 0..n (n + 1 tokens: the KV of the last committed
 * token and of d_0..d_{n-1}) are copied, for all layers and both K and V, to logical
 * positions L..L+n of the row's own blocks. New blocks come from the top of the free
 * stack, rows in ascending order, before any block is pushed; then every provisional
 * block is pushed back in row order. All-or-nothing: if any row is invalid or the
 * stack is short, nothing changes and *status receives the error bits. Validation
 * checks, per row: n in [0, K]; L >= 0 and ceil((L+n+1)/bs) <= max_blocks; the
 * partly filled tail block (index L/bs when L % bs != 0) is a valid id; the
 * entries the commit fills are -1; the provisional blocks of the kept slots are valid
 * and every provisional id >= 0 is < num_blocks. Globally: 0 <= *free_top <=
 * num_blocks and covers the new blocks, the popped ids are valid, and the pushes fit.
 * Only the accepted bytes move. Blocks freed by the call must not be reused until
 * the stream passes it.
 */
int kv_commit_rollback(int32_t* block_table, int32_t* seq_lens, const int32_t* num_accepted,
                       int32_t* prov_blocks, void* kv_pool, int num_blocks, int num_layers,
                       int num_kv_heads, int head_dim, int kv_elem_bytes, int block_size, int B,
                       int K, int max_blocks, int P, int32_t* free_stack, int32_t* free_top,
                       int32_t* status, void* stream, const int32_t* slot_map);

/*
 * kv_commit_inplace - commit for the in-place KV layout ([L] "Rolling back the KV
 * cache": keep the physical cache and truncate a logical length).
 *
 * Layout: before the verify step the caller appended the K+1 provisional slots
 * at logical positions L_b .. L_b + K of each row's OWN blocks (block_table
 * entries [0, ceil((L_b + K + 1) / block_size)) valid). The commit sets the
 * length to L_b + n_b + 1 and frees every block that then holds no position
 * below it: block indices ceil((L_b + n_b + 1) / bs) .. ceil((L_b + K + 1) / bs) - 1
 * are pushed onto the free stack (rows ascending, indices ascending) and set to
 * -1. No KV byte moves, so no pool pointer is needed.
 *   block_table [B, max_blocks] int32; seq_lens [B] int32 (L_b, becomes L_b + n_b + 1);
 *   num_accepted [B] int32 in [0, K]; free_stack [num_blocks] int32 with live
 *   entries [0, *free_top); status REQUIRED [1] int32: 0, or the SPEC_DERR_* bits
 *   that stopped the call (then nothing changed: all-or-nothing).
 * Device errors: SPEC_DERR_BAD_ACCEPT (n outside [0, K]), SPEC_DERR_BAD_LENGTH
 * (L < 0 or L + K + 1 beyond max_blocks * block_size), SPEC_DERR_BAD_BLOCK (a
 * table entry holding a provisional slot outside [0, num_blocks), or the pushes
 * would overflow the stack). Host errors: SPEC_EINVAL (null pointer, sizes,
 * K outside [0, 31]).
 */
int kv_commit_inplace(int32_t* block_table, int32_t* seq_lens, const int32_t* num_accepted,
                      int num_blocks, int block_size, int B, int K, int max_blocks,
                      int32_t* free_stack, int32_t* free_top, int32_t* status, void* stream);

/*
 * kv_evict_provisional - preemption of rows in the in-place layout ([S]: a
 * preempted request's provisional KV is evicted): as kv_commit_inplace with
 * every row's length reset to L_b (all K+1 provisional slots discarded).
 */
int kv_evict_provisional(int32_t* block_table, int32_t* seq_lens, int num_blocks,
                         int block_size, int B, int K, int max_blocks, int32_t* free_stack,
                         int32_t* free_top, int32_t* status, void* stream);

/*
 * spec_selftest_ex2 - diagnostic: the maximum relative error of the hardware
 * base-2 exponential over every fp32 argument in [lo, hi] (-126 <= lo <= hi <= 127),
 * measured against fp64 exp2 and written to the device double *out_max_rel.
 * The sampler's certification assumes this maximum stays below its built-in
 * bound on [-126, 127]; tests re-measure it on the GPU in use.
 */
int spec_selftest_ex2(float lo, float hi, double* out_max_rel, void* stream);

/* Human-readable text of a status code (static string). */
const char* spec_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int spec_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
