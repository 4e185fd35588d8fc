/*
 * flp.h - C ABI of the fused linear log-prob / cross-entropy LM head for
 * GB300 (sm_103a).
 *
 * Problem (Liger-Kernel v0.8.3 test/transformers page, the native SM100 fused
 * scaled linear cross-entropy commit, section "Summary": the classifier GEMM
 * fused with NLL/LSE and optional entropy; "Chunked Triton GRPO loss" of the
 * Liger-Kernel pull request 1294 page: the lm_head fused into the loss with an
 * online logsumexp so that the (N, V) logits are never materialised):
 *
 *   X  : bf16 [M, H], row-major, contiguous   (hidden states)
 *   W  : bf16 [V, H], row-major, contiguous   (classifier / lm_head weight,
 *                                              the nn.Linear layout)
 *   y  : int64 [M]                            (targets, ignore_index allowed)
 *   s  : fp32                                 (logit scale, 1/temperature)
 *
 *   z_ij      = s * sum_k X_ik W_jk   (fp32 accumulation; never stored in HBM)
 *   lse_i     = log sum_j exp(z_ij)
 *   logprob_i = z_{i,y_i} - lse_i
 *   entropy_i = lse_i - sum_j p_ij z_ij,   p_ij = exp(z_ij - lse_i)
 *
 * Backward (same Liger-Kernel pages: "Implementation > Backward" of the native
 * commit, "Kernel design notes" of pull request 1294): the logits are
 * recomputed tile by tile,
 *
 *   dZ_ij = s * [ g_lp_i (1[j = y_i] - p_ij) + g_ent_i p_ij (sum_k p_ik z_ik - z_ij) ]
 *
 * is rounded to bf16, and contracted into dX = dZ W and dW = dZ^T X with fp32
 * accumulation.
 *
 * Conventions shared by every entry point
 *  - Device pointers are CUDA device addresses owned by the caller; the library
 *    allocates no device memory and keeps no state between calls beyond cached
 *    device attributes.  Every call is asynchronous on `stream` (a
 *    cudaStream_t passed as void*, NULL for the legacy default stream) and
 *    launches only on the device that is current on the calling thread.
 *  - Argument errors are returned synchronously before anything is launched.
 *    Required: every pointer 16-byte aligned; H % 8 == 0 (row pitch of a TMA
 *    tensor, else FLP_ERR_UNSUPPORTED); M >= 0 (M == 0 is a no-op); V >= 1;
 *    workspace large enough (else FLP_ERR_WORKSPACE).
 *  - A row whose target equals ignore_index has logprob = 0, entropy = 0 and a
 *    zero gradient row; its lse is still written.  A target outside [0, V)
 *    that is not ignore_index yields logprob = NaN for that row and sets
 *    FLP_ERR_BAD_TARGET in the workspace's error word (read it with
 *    flp_get_error); the call itself still returns FLP_OK because the hot path
 *    never synchronises.
 *  - The workspace is caller-owned device memory of at least the queried size.
 *    Its contents need no initialisation; a call owns it until the work it
 *    queued on `stream` has finished.  Calls that run concurrently must use
 *    distinct workspaces.
 *  - Results are deterministic: no floating-point atomics are used, so two
 *    identical calls produce bit-identical outputs.
 */
#ifndef FLP_H
#define FLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FLP_OK = 0,
    FLP_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, bad flag */
    FLP_ERR_UNSUPPORTED = 2, /* shape or device the kernels do not handle (H % 8 != 0,
                                not an sm_103 device, size beyond int32 tiling) */
    FLP_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than required */
    FLP_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed; see flp_last_error_message */
    FLP_ERR_BAD_TARGET = 5,  /* (error word) a target outside [0, V) that is not ignore_index */
    FLP_ERR_TIMEOUT = 6      /* (error word) a kernel's bounded wait expired; its outputs are invalid */
} flp_status;

typedef enum { FLP_F32 = 0, FLP_BF16 = 1 } flp_dtype;

/*
 * Workspace sizes, in bytes, for the given problem on the current device
 * (the Liger-Kernel native commit's "Summary" lists reusable workspace
 * configuration and query APIs).
 *   fwd_bytes : needed by flp_forward (per-split raw partials and the target
 *               logits; the SkyRL page "perf(megatron): autotune fused LM-head
 *               Triton kernels", section "Correctness", keeps raw and final
 *               results in separate buffers, and so does this library).
 *   bwd_bytes : needed by flp_backward with its default row waves of up to
 *               8192 rows (all M rows when M <= 8192); one wave's bf16 dZ,
 *               [wave rows, ceil(V/256)*256], dominates, beside a few KiB of
 *               tile counters.  The native commit's "Memory" section reports
 *               the same kind of reusable workspace, and pull request 1294's
 *               "Kernel design notes" a reusable per-chunk grad_logits buffer.
 * Either output pointer may be NULL.  The same buffer may serve both calls.
 * Returns FLP_ERR_INVALID_ARG for negative sizes, FLP_ERR_CUDA if the device
 * cannot be queried (FLP_ERR_UNSUPPORTED if it is not an sm_103 device).
 */
flp_status flp_workspace_query(int64_t M, int64_t H, int64_t V, int compute_entropy,
                               size_t* fwd_bytes, size_t* bwd_bytes);

/*
 * flp_workspace_query with the backward's wave size chosen by the caller:
 * bwd_bytes is what flp_backward needs to process the rows in waves of
 * `chunk_rows` rows (rounded up to a multiple of 128, at most M;
 * chunk_rows <= 0 selects the default of flp_workspace_query).  A smaller
 * wave trades speed for a smaller workspace; below 2048-row waves
 * flp_backward runs the vocabulary-split schedule instead when the same bytes
 * also hold its fp32 dX scratch (see flp_backward_ex).  Errors as
 * flp_workspace_query.
 */
flp_status flp_workspace_query_ex(int64_t M, int64_t H, int64_t V, int compute_entropy,
                                  int64_t chunk_rows, size_t* fwd_bytes, size_t* bwd_bytes);

/*
 * Forward: writes logprob[M], lse[M] and (when compute_entropy != 0)
 * entropy[M], all fp32 device arrays.  entropy must be NULL when
 * compute_entropy == 0 and non-NULL otherwise (the SkyRL page's "Overview":
 * compute_entropy gates the entropy buffers and kernel work).
 * Two kernels run on `stream`: the fused tcgen05 GEMM + online
 * max / sum-exp / target / entropy epilogue writing raw per-split partials to
 * the workspace, then the merge of those partials into the outputs.  If a
 * bounded wait of the first kernel runs out (FLP_ERR_TIMEOUT in the error
 * word), the merge writes NaN to every output row.
 */
flp_status flp_forward(const void* X, const void* W, const int64_t* targets, int64_t M,
                       int64_t H, int64_t V, int64_t ignore_index, float scale,
                       int compute_entropy, float* logprob, float* lse, float* entropy,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: given the forward's lse (and entropy when compute_entropy != 0),
 * writes dX [M, H] (dtype dX_dtype, overwritten) and dW [V, H] (dtype
 * dW_dtype; overwritten, or added to when accumulate_dW != 0).  An FLP_F32 dW
 * accumulates in fp32 across waves.  An FLP_BF16 dW is written once, rounded
 * from the fp32 accumulator, so it needs the whole backward in one wave (a
 * workspace that holds all M rows of dZ) and no accumulate_dW; otherwise the
 * call returns FLP_ERR_UNSUPPORTED before launching anything.
 *   grad_logprob, grad_entropy : fp32 [M] upstream gradients of logprob and
 *       entropy; NULL means zero.  grad_entropy is ignored when
 *       compute_entropy == 0.  For a mean NLL loss over N valid rows pass
 *       grad_logprob = -1/N on every row.
 * Rows are processed in waves of as many rows as the workspace holds (at most
 * M, at least 128): each wave recomputes its logits tiles, writes bf16 dZ to
 * the workspace, and runs the dX and dW contractions; dW accumulates in fp32
 * across waves in a fixed order.  flp_backward picks the schedule
 * (FLP_BWD_AUTO of flp_backward_ex).
 */
flp_status flp_backward(const void* X, const void* W, const int64_t* targets, int64_t M,
                        int64_t H, int64_t V, int64_t ignore_index, float scale,
                        int compute_entropy, const float* lse, const float* entropy,
                        const float* grad_logprob, const float* grad_entropy, void* dX,
                        flp_dtype dX_dtype, void* dW, flp_dtype dW_dtype, int accumulate_dW,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * How the backward's tiles are scheduled (the Liger-Kernel native commit,
 * "Implementation > Backward": persistent kernels over token waves).
 *   FLP_BWD_SPLIT : per wave, one launch of the wave's dZ tiles, then one
 *                   launch of its dX and dW tiles.  Waves may be any multiple
 *                   of 128 rows.
 *   FLP_BWD_FUSED : one persistent launch for every wave: dX and dW tiles
 *                   start as soon as the dZ tiles they read are stored (tile
 *                   counters in the workspace), most dW tiles run interleaved
 *                   with the dZ sweep while their dZ column is still in L2,
 *                   and a wave's last dW tiles overlap the next wave's dZ
 *                   tiles.  With more than one wave, waves are multiples of
 *                   256 rows.
 *   FLP_BWD_VSPLIT: all rows in one wave and the vocabulary in chunks of as
 *                   many columns as the workspace holds after an fp32 [M, H]
 *                   dX scratch: per chunk, one launch of its dZ tiles and one
 *                   of its dX and dW tiles.  dX accumulates over the chunks
 *                   in fp32 (in the scratch when dX is bf16, rounded once at
 *                   the end), and every dW tile is written once with K = all
 *                   rows, so a small workspace keeps long dW contractions and
 *                   a bf16 dW stays possible.  dW is bit-identical to a
 *                   one-wave run of the other schedules; dX differs from it
 *                   by the fp32 summation order over the chunks.
 *   FLP_BWD_AUTO  : the faster one on GB300: FLP_BWD_SPLIT when its waves
 *                   hold all rows or at least 2048 rows, else FLP_BWD_VSPLIT
 *                   when the workspace allows it (else FLP_BWD_SPLIT).  The
 *                   fused launch keeps 256 x 256 dZ and dW tiles (its
 *                   dependency counters count 256-column tiles) where the
 *                   split schedule runs 256 x 512 ones, and measured ~7%
 *                   slower per headline step; with the same tile shapes in
 *                   both schedules it was 0.6-2% slower at every shape
 *                   measured.
 * The split and fused schedules compute every output tile with the same
 * instructions in the same order: their results are bit-identical.
 */
typedef enum { FLP_BWD_AUTO = 0, FLP_BWD_SPLIT = 1, FLP_BWD_FUSED = 2, FLP_BWD_VSPLIT = 3 } flp_bwd_schedule;

/*
 * flp_backward with an explicit schedule.  FLP_BWD_FUSED returns
 * FLP_ERR_UNSUPPORTED when the workspace holds fewer than 256 rows of dZ but
 * not all M rows; other arguments and errors are those of flp_backward.
 */
flp_status flp_backward_ex(const void* X, const void* W, const int64_t* targets, int64_t M,
                           int64_t H, int64_t V, int64_t ignore_index, float scale,
                           int compute_entropy, const float* lse, const float* entropy,
                           const float* grad_logprob, const float* grad_entropy, void* dX,
                           flp_dtype dX_dtype, void* dW, flp_dtype dW_dtype, int accumulate_dW,
                           void* workspace, size_t workspace_bytes, flp_bwd_schedule schedule,
                           void* stream);

/*
 * The wave size, wave count and schedule (FLP_BWD_SPLIT, FLP_BWD_FUSED or
 * FLP_BWD_VSPLIT) that flp_backward_ex would use for this problem, workspace
 * size and requested schedule; for FLP_BWD_VSPLIT *waves counts vocabulary
 * chunks.  Host arithmetic only: touches no device.  Any output
 * pointer may be NULL.  Returns FLP_ERR_WORKSPACE / FLP_ERR_UNSUPPORTED
 * exactly when the backward call would.
 */
flp_status flp_backward_plan(int64_t M, int64_t H, int64_t V, size_t workspace_bytes,
                             flp_bwd_schedule schedule, int64_t* wave_rows, int64_t* waves,
                             flp_bwd_schedule* schedule_used);

/*
 * The backward's tile schedule, for inspection (a diagnostic; host arithmetic
 * only, touches no device): the units that flp_backward_ex would hand out, in
 * ticket order over its launches, for `pairs` resident CTA pairs.  Entry n is
 * units[5n .. 5n+4] = (launch, kind, wave, a, b), kind 0 = dZ tile (a = row
 * tile of the wave, b = vocabulary tile), 1 = dX tile (a = row tile, b =
 * hidden tile), 2 = dW tile (a = vocabulary tile, b = hidden tile), 3 = wide
 * dX tile (a = row tile, b = 512-column hidden tile: the hidden tiles 2b and
 * 2b + 1), 4 = wide dZ tile (a = row tile, b = its first vocabulary tile: the
 * vocabulary tiles b and b + 1; one whose second half lies past the launch's
 * vocabulary is listed as the dZ tile b, kind 0), 5 = wide dW tile (a =
 * vocabulary tile, b = 512-column hidden tile: the hidden tiles 2b and
 * 2b + 1); tiles are 256 x 256 except the wide ones.  At most `capacity` entries are written; *count receives the
 * total.  units may be NULL to query the count.
 */
flp_status flp_backward_schedule(int64_t M, int64_t H, int64_t V, size_t workspace_bytes,
                                 flp_bwd_schedule schedule, int pairs, int32_t* units,
                                 int64_t capacity, int64_t* count);

/*
 * Forward that allocates nothing and takes no workspace.  The pages have no
 * counterpart; it exists for callers that cannot call cudaMalloc and have no
 * workspace to hand: code running inside a host framework that owns every
 * device allocation and gives its plugins no allocator, or latency-critical
 * loops where the implicit device synchronisation of cudaMalloc/cudaFree is
 * not acceptable.  Arguments and outputs are those of flp_forward; the
 * per-split partials and the error word live instead in one file-scope
 * device array of FLP_STATIC_SCRATCH_BYTES (16 MiB) that every GPU which
 * loads this library holds until the process exits.
 *  - It takes the fastest vocabulary-split plan whose scratch fits that size
 *    (flp_forward's own plan when its fwd_bytes fit, with the same results
 *    bit for bit; otherwise fewer splits, whose merged results can differ from
 *    flp_forward's in the last bits).  Problems that do not fit even with one
 *    split are rejected with FLP_ERR_UNSUPPORTED before any launch.
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress, with the device current); make that first
 *    call before any stream capture.  No cudaMalloc, cudaFree or allocating
 *    library routine is ever called.
 *  - Every call, on any stream, shares the one array and it keeps the last
 *    call's contents (each call clears its error word first): calls that
 *    overlap on the GPU race and corrupt each other's results.
 *  - Out-of-range targets still give logprob = NaN; the error word of this
 *    array is not readable through flp_get_error.  If a bounded wait of the
 *    forward kernel ever runs out, the merge writes NaN to every output row,
 *    so a failed call cannot pass stale values from the array for results.
 */
#define FLP_STATIC_SCRATCH_BYTES (16u << 20)
flp_status flp_forward_noalloc(const void* X, const void* W, const int64_t* targets, int64_t M,
                               int64_t H, int64_t V, int64_t ignore_index, float scale,
                               int compute_entropy, float* logprob, float* lse, float* entropy,
                               void* stream);

/*
 * Loss heads on the forward's per-row log-probs (the chunked GRPO page,
 * "Chunked Triton GRPO loss": a loss on top of the lm_head's per-token
 * log-probs).  With N = the number of rows whose target is not ignore_index:
 *   FLP_LOSS_NLL_MEAN           loss = -(1/N) sum_i lp_i
 *   FLP_LOSS_NLL_SUM            loss = -sum_i lp_i  (token-sum reduction;
 *                               grad_logprob = -1 on every valid row)
 *   FLP_LOSS_CLIPPED_SURROGATE  r_i = exp(lp_i - old_i),
 *       loss = (1/N) sum_i [ -min(r_i A_i, clip(r_i, 1 - eps_low, 1 + eps_high) A_i)
 *                            + beta (exp(ref_i - lp_i) - (ref_i - lp_i) - 1) ]
 *       (token-level ratio, two-sided clip, k3 KL estimator against a
 *       reference policy when ref_logprob != NULL).
 * All arrays are fp32 [M] device arrays: old_logprob and advantage are
 * required for the clipped surrogate and ignored otherwise; per_token_loss
 * (the bracketed terms, 0 on ignored rows) and grad_logprob (d loss / d lp_i,
 * the upstream gradient to hand to flp_backward) may be NULL; loss is one
 * fp32 on the device.  One block with fixed-order fp64 reductions:
 * deterministic.  N = 0 gives loss 0 and zero gradients.
 */
typedef enum { FLP_LOSS_NLL_MEAN = 1, FLP_LOSS_CLIPPED_SURROGATE = 2, FLP_LOSS_NLL_SUM = 3 } flp_loss_kind;
flp_status flp_loss(const float* logprob, const int64_t* targets, int64_t M, int64_t ignore_index,
                    int kind, const float* old_logprob, const float* advantage,
                    const float* ref_logprob, float eps_low, float eps_high, float beta,
                    float* per_token_loss, float* grad_logprob, float* loss, void* stream);

/*
 * Clipped-surrogate policy loss over sequences (the chunked GRPO page: its
 * "Setup" runs loss_type="dapo" with importance_sampling_level="sequence" and
 * num_items_in_batch, its "Correctness" section covers the grpo / bnpo /
 * dr_grpo / dapo aggregations with token- and sequence-level ratios).  The
 * page names these options without defining them; this library reads them so:
 *   seq_offsets : int64 [num_seqs + 1] device array; rows [off[b], off[b+1])
 *                 form sequence b (ranges are clamped to [0, M); they must not
 *                 overlap).  NULL: one sequence of all M rows.  A row is a
 *                 token of the loss when its target is not ignore_index; n_b
 *                 counts the tokens of sequence b, N all of them.
 *   is_level    : FLP_IS_TOKEN     log r_t = lp_t - old_t
 *                 FLP_IS_SEQUENCE  log r_t = (1/n_b) sum_{u in b} (lp_u - old_u),
 *                                  shared by every token of b
 *   term_t      = -min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t)
 *                 + beta (exp(ref_t - lp_t) - (ref_t - lp_t) - 1)  (when ref_logprob != NULL)
 *   aggregation : FLP_AGG_TOKEN_MEAN     loss = (1/N) sum_t term_t            (bnpo)
 *                 FLP_AGG_SEQUENCE_MEAN  loss = (1/B) sum_b (1/max(n_b,1)) sum_{t in b} term_t (grpo)
 *                 FLP_AGG_SUM_OVER       loss = (1/D) sum_t term_t, D = normalizer when > 0
 *                                        (dapo: num_items_in_batch, the token count of the
 *                                        whole global batch; dr_grpo: B x the longest
 *                                        completion), else D = N
 * Outputs as flp_loss: per_token_loss (term_t, 0 on rows that are not
 * tokens) and grad_logprob (d loss / d lp_t, the upstream gradient for
 * flp_backward; with a sequence-level ratio it includes every term of the
 * sequence through log r_b) may be NULL; loss is one fp32 on the device.
 * old_logprob and advantage (per row: broadcast a per-sequence advantage) are
 * required.  One block, fp64 arithmetic, fixed-order reductions:
 * deterministic.  FLP_LOSS_CLIPPED_SURROGATE of flp_loss is the token-level
 * ratio with FLP_AGG_TOKEN_MEAN.
 */
typedef enum { FLP_IS_TOKEN = 0, FLP_IS_SEQUENCE = 1 } flp_is_level;
typedef enum { FLP_AGG_TOKEN_MEAN = 0, FLP_AGG_SEQUENCE_MEAN = 1, FLP_AGG_SUM_OVER = 2 } flp_loss_aggregation;
flp_status flp_policy_loss(const float* logprob, const int64_t* targets, int64_t M,
                           int64_t ignore_index, const int64_t* seq_offsets, int64_t num_seqs,
                           const float* old_logprob, const float* advantage,
                           const float* ref_logprob, float eps_low, float eps_high, float beta,
                           int is_level, int aggregation, double normalizer,
                           float* per_token_loss, float* grad_logprob, float* loss, void* stream);

/*
 * Synchronises `stream`, then reads and returns the workspace's error word
 * (FLP_OK, FLP_ERR_BAD_TARGET or FLP_ERR_TIMEOUT) written by the most recent
 * flp_forward / flp_backward that used this workspace.  Each of those calls
 * clears the word when it starts.  Returns FLP_ERR_CUDA if the copy fails.
 */
flp_status flp_get_error(const void* workspace, void* stream);

/*
 * Optional instrumentation for benchmarks and profiling.  After this call the
 * calling thread's flp_forward / flp_backward record events[2k] immediately
 * before and events[2k+1] immediately after kernel phase k, on the call's
 * stream:
 *   k = 0  forward tile kernel          k = 1  split merge
 *   k = 2  FLP_BWD_SPLIT: the first wave's dZ launch;
 *          FLP_BWD_FUSED: the one backward launch (every wave)
 *   k = 3  FLP_BWD_SPLIT: the first wave's dX and dW launch (not recorded
 *          by FLP_BWD_FUSED)
 *   k = 4  reserved (never recorded)
 * `events` holds `count` (<= 10) caller-created cudaEvent_t handles passed as
 * void*; NULL entries are skipped.  events == NULL or count == 0 turns the
 * instrumentation off.  The array is copied; the events stay caller-owned.
 * Returns FLP_ERR_INVALID_ARG when count is outside [0, 10].
 */
flp_status flp_set_phase_events(void* const* events, int count);

/*
 * Self-test of the kernels' bounded waits (a diagnostic; the pages have no
 * counterpart).  Runs the forward (tile kernel, then the split merge) on a
 * small internal problem (M = 256, H = 256, V = 512, all-zero inputs, targets
 * 0) laid out in `workspace` (caller-owned device memory of at least
 * FLP_SELFTEST_WORKSPACE_BYTES).  With stall_after >= 0 the TMA producers
 * stop after that many pipeline stages, so the MMA issuer waits for data that
 * never arrives: every wait gives up after wait_limit_ns, the kernel records
 * FLP_ERR_TIMEOUT in the error word, lets its copies and MMAs in flight
 * finish, frees its TMEM and returns; nothing faults and the context stays
 * usable.  The merge then finds the timeout bit and writes NaN to every
 * output.  With stall_after < 0 the same launches run normally (every row:
 * lse = entropy = log 512, logprob = -log 512).  The outputs, fp32 logprob,
 * lse and entropy of the 256 rows one after the other, are left in the
 * workspace at byte offset FLP_SELFTEST_OUTPUT_OFFSET.  Synchronises `stream`
 * and returns the error word (FLP_ERR_TIMEOUT, or FLP_OK), or an argument /
 * CUDA error.
 */
#define FLP_SELFTEST_WORKSPACE_BYTES (1u << 20)
#define FLP_SELFTEST_OUTPUT_OFFSET (768u << 10)
flp_status flp_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int stall_after,
                                     int64_t wait_limit_ns, void* stream);

/*
 * Self-test of the fused backward schedule's dependency waits (a diagnostic;
 * the pages have no counterpart).  Runs one fused-schedule launch of the
 * backward kernel on a small internal all-zero problem (M = H = V = 256)
 * laid out in `workspace` (at least FLP_SELFTEST_WORKSPACE_BYTES).  With
 * broken != 0 the schedule holds only the dX tile, whose wait for its dZ tile
 * can never be met: the wait gives up after wait_limit_ns, the kernel records
 * FLP_ERR_TIMEOUT, winds down (bounded) and returns; nothing faults and the
 * context stays usable.  With broken == 0 the full schedule runs normally.
 * Synchronises `stream` and returns the error word (FLP_ERR_TIMEOUT or
 * FLP_OK), or an argument / CUDA error.
 */
flp_status flp_selftest_dependency_timeout(void* workspace, size_t workspace_bytes, int broken,
                                           int64_t wait_limit_ns, void* stream);

/*
 * The same self-test for the backward's dZ kernel (the split and
 * vocabulary-split schedules' dZ launch; a diagnostic, the pages have no
 * counterpart): one 256 x 512 dZ tile of a small internal all-zero problem
 * (M = 256, H = 256, V = 512) laid out in `workspace` (at least
 * FLP_SELFTEST_WORKSPACE_BYTES).  With stall_after >= 0 its TMA producers
 * stop after that many pipeline stages: the MMA issuer's wait gives up after
 * wait_limit_ns, the kernel records FLP_ERR_TIMEOUT, its epilogue warps stop
 * together (a vote before any store barrier), it winds down (bounded) and
 * returns; nothing faults and the context stays usable.  With
 * stall_after < 0 the tile runs normally.  Synchronises `stream` and returns
 * the error word (FLP_ERR_TIMEOUT or FLP_OK), or an argument / CUDA error.
 */
flp_status flp_selftest_dz_wait_timeout(void* workspace, size_t workspace_bytes, int stall_after,
                                        int64_t wait_limit_ns, void* stream);

/* Static description of a status code. */
const char* flp_status_string(flp_status status);

/* Text of the last FLP_ERR_CUDA / FLP_ERR_UNSUPPORTED on the calling thread. */
const char* flp_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* FLP_H */
