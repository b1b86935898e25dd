/*
 * gbce.h - C ABI of the GB300 fused softmax cross-entropy library
 * (libgbce.so, built for sm_103a).
 *
 * One call computes, for every row i of a (rows, V) logit matrix x, the
 * cross-entropy loss against an integer target, and (optionally) writes the
 * gradient of the reduced loss in place over x. Backward then only scales
 * the stored gradient by grad_output.
 *
 * Definitions followed (page title, section):
 *  - "Kernel Profile: CrossEntropy (Tier 3 - Fused/Complex)" (Liger-Kernel),
 *    §Forward Pass: inputs _input (B*T, V), target (B*T,), weight (V,) or
 *    none, ignore_index, label_smoothing, reduction "mean" | "sum" | "none",
 *    softcap; outputs loss (scalar, or (B*T,) for "none"), z_loss,
 *    token_accuracy, predicted_tokens; exp and log run in fp32.
 *    §Backward Pass: the gradient is computed during the forward and stored
 *    in the _input tensor; backward scales it by grad_output.
 *    §Module Parameters: ignore_index = -100 by default, lse_square_scale.
 *    §Key Patterns: max-shifted log-sum-exp; the loss combines CE, the
 *    label-smoothing loss and the z-loss, each contributing to the gradient.
 *  - tenstorrent/tt-mlir pull request #9324 "[tt-crank] fuse cross entropy
 *    onto the ttml cross_entropy_fw/bw composites", review comments: the
 *    mean divides by total_weight; a batch whose rows are all ignored keeps
 *    the NaN forward loss and gets exactly zero gradients.
 *
 * Per row, with z = softcap(x) = s * tanh(x / s) (s > 0) or z = x,
 * lse = log sum_j exp(z_j), p = exp(z - lse), target t, class weights w
 * (all 1 when weight is NULL), W = sum_j w_j, eps = label_smoothing and
 * lam = lse_square_scale:
 *
 *   loss_i = (1 - eps) * w_t * (lse - z_t)
 *          + (eps / V) * sum_j w_j * (lse - z_j)
 *          + lam * lse^2                         (z_loss_i = lam * lse^2)
 *   dlogits_ik = scale * [ (1 - eps) * w_t * (p_k - [k == t])
 *                        + (eps / V) * (W * p_k - w_k)
 *                        + 2 * lam * lse * p_k ] * dz_k/dx_k
 *
 * with scale = 1 / D for "mean" and 1 otherwise, D = sum of w_{t_i} over the
 * rows whose target is not ignore_index. A row whose target equals
 * ignore_index has loss 0, z_loss 0, predicted token -1 and a gradient of
 * exact +0; its logits are never read. Reductions: "sum" adds the rows,
 * "mean" divides the sums by D (so a batch with every row ignored gives a
 * NaN loss, NaN z_loss and zero gradients), "none" returns per-row values.
 * Accuracy is n_correct / n_valid for "sum"/"mean" (NaN with no valid row)
 * and a 0/1 value per row for "none"; a row is correct when its argmax
 * (over the raw logits, lowest index on ties) equals its target.
 *
 * Arithmetic: fp32 in registers for every input dtype (fp32, bf16, fp16);
 * gradients are rounded to nearest-even into the logit dtype (fp16
 * gradients below 2^-24 in magnitude round to zero or a subnormal). Partial sums of the scalar
 * outputs are combined in a fixed order, so results are run-to-run
 * deterministic.
 *
 * Threading and streams: every call is asynchronous on `stream` (NULL is
 * the legacy default stream). All pointers are device pointers owned by
 * the caller. The library keeps a small scratch area per (device, stream),
 * allocated with cudaMalloc on the first call for that pair and kept until
 * the process exits; make that first call outside any CUDA graph capture.
 * Calls on the same stream are ordered; calls on different streams use
 * different scratch areas.
 */
#ifndef GBCE_H
#define GBCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* ce_stream_t;

typedef enum {
    CE_OK = 0,
    CE_ERR_INVALID_ARG = 1,   /* argument check failed; nothing was enqueued */
    CE_ERR_UNSUPPORTED = 2,   /* valid arguments outside what is implemented */
    CE_ERR_CUDA = 3,          /* a CUDA runtime call failed (see ce_last_error) */
    CE_ERR_TARGET_RANGE = 4,  /* the device saw a target outside [0, V) that is not ignore_index */
    CE_ERR_TIMEOUT = 5        /* a bounded device wait gave up; that call's outputs are invalid */
} ce_status;

typedef enum { CE_F32 = 0, CE_BF16 = 1, CE_F16 = 2 } ce_dtype;

typedef enum { CE_RED_NONE = 0, CE_RED_SUM = 1, CE_RED_MEAN = 2 } ce_reduction;

enum {
    CE_FLAG_GRAD = 1,        /* write dlogits in place over logits */
    CE_FLAG_Z_LOSS = 2,      /* write z_loss */
    CE_FLAG_ACC = 4,         /* write token accuracy to acc */
    CE_FLAG_PRED = 8,        /* write predicted tokens to pred */
    CE_FLAG_TARGET_I64 = 16  /* target is int64 (default int32) */
};

/*
 * ce_fwd - fused forward (and, with CE_FLAG_GRAD, the in-forward gradient).
 *
 * logits       [rows, V] row-major, dtype `dtype` (CE_F32, CE_BF16 or CE_F16). With
 *              CE_FLAG_GRAD it is overwritten by dlogits (d loss / d logits
 *              of the reduced loss; for "none", of the sum of the row
 *              losses). The fast path needs a 16-byte aligned base and
 *              V * sizeof(dtype) a multiple of 16; other shapes take a
 *              slower general path with the same results.
 * rows, V      rows >= 0, 1 <= V < 2^31.
 * target       [rows] int32 (int64 with CE_FLAG_TARGET_I64). A value equal
 *              to ignore_index marks an ignored row. A value outside [0, V)
 *              that is not ignore_index is an error: that row is treated as
 *              ignored and CE_ERR_TARGET_RANGE is recorded for
 *              ce_device_status.
 * weight       [V] fp32 class weights, or NULL for all ones.
 * label_smoothing   in [0, 1].
 * lse_square_scale  finite; 0 turns the z-loss term off.
 * softcap      0 turns softcapping off; > 0 is the cap s; negative or
 *              non-finite values are invalid.
 * reduction    CE_RED_NONE, CE_RED_SUM or CE_RED_MEAN.
 * flags        CE_FLAG_* bits.
 * loss         fp32, [rows] for CE_RED_NONE else [1]. Required.
 * z_loss       same shape as loss; required with CE_FLAG_Z_LOSS.
 * acc          same shape as loss; required with CE_FLAG_ACC.
 * pred         [rows] int64 (-1 on ignored rows); required with CE_FLAG_PRED.
 * stream       CUDA stream of the launch.
 *
 * rows == 0: "mean" writes NaN to loss (and z_loss), "sum" writes 0, acc
 * gets NaN. Returns CE_OK when the work was enqueued; CE_ERR_INVALID_ARG or
 * CE_ERR_UNSUPPORTED with nothing enqueued; CE_ERR_CUDA on a failed launch.
 */
ce_status ce_fwd(void* logits, int dtype, int64_t rows, int64_t V,
                 const void* target, const float* weight, int64_t ignore_index,
                 float label_smoothing, float lse_square_scale, float softcap,
                 int reduction, uint32_t flags, float* loss, float* z_loss,
                 float* acc, int64_t* pred, ce_stream_t stream);

/*
 * ce_fwd_noalloc - ce_fwd for callers that cannot allocate device memory.
 *
 * The method has no counterpart for this call: it exists for code that may
 * not call cudaMalloc, such as an allocator's own callbacks, a memory-capped
 * sandbox, or a framework that forbids allocations once it has started.
 * ce_fwd keeps a small scratch area per (device, stream) that it allocates on
 * first use; this call instead uses one fixed device array compiled into the
 * library (about 64 KB, held by every GPU that loads the library until the
 * process exits) and allocates nothing.
 *
 * Arguments, outputs and results are those of ce_fwd. Differences:
 *  - The scratch holds 2048 partial-sum slots, one per CTA (or cluster) of
 *    the launch; a launch that would need more returns CE_ERR_UNSUPPORTED
 *    with nothing enqueued, and ce_last_error names the number. (Every
 *    launch plan of this library is capped at 8 slots per SM, 1216 on a
 *    GB300's 152 SMs, so this happens only on a GPU with more than 256
 *    SMs.)
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call, on every stream, shares the same array. Each call clears
 *    the part that must start at zero (the epilogue's ticket), but calls
 *    that overlap on the GPU (different streams, or concurrent host
 *    threads) race on it; order them on one stream or synchronise between
 *    them.
 *  - Device-detected errors (a target outside [0, V), a bounded wait that
 *    ran out) go to the array's own sticky status word, which
 *    ce_noalloc_status reads and clears; ce_device_status does not see it.
 *  - Test hook, read at each call: GBCE_TEST_NOALLOC_SLOTS=n (1 <= n <
 *    2048) lowers the usable slots to n, so that the refusal above can be
 *    exercised on any GPU.
 */
ce_status ce_fwd_noalloc(void* logits, int dtype, int64_t rows, int64_t V,
                         const void* target, const float* weight, int64_t ignore_index,
                         float label_smoothing, float lse_square_scale, float softcap,
                         int reduction, uint32_t flags, float* loss, float* z_loss,
                         float* acc, int64_t* pred, ce_stream_t stream);

/*
 * ce_noalloc_status - the device-detected errors of ce_fwd_noalloc calls.
 *
 * Like ce_device_status, but for the fixed array ce_fwd_noalloc uses (the
 * method has no counterpart for it either). Synchronises `stream`, copies
 * the array's status word of the current device into a host variable,
 * clears it, and returns CE_ERR_TIMEOUT or CE_ERR_TARGET_RANGE if any
 * ce_fwd_noalloc call since the last read recorded one (the word is shared
 * by every stream), else CE_OK. Allocates nothing; CE_ERR_CUDA if a copy
 * or the synchronisation fails.
 */
ce_status ce_noalloc_status(ce_stream_t stream);

/*
 * ce_count - counts of one shard of rows, for a "mean" over a batch whose
 * rows are split across calls or GPUs (the mean divides by D, the sum of
 * w[t_i] over the rows that take part: "Kernel Profile: CrossEntropy",
 * §Forward Pass, reductions; tt-mlir pull request #9324 review comments,
 * total_weight).
 *
 * target, weight, rows, V, ignore_index, flags (only CE_FLAG_TARGET_I64)
 *              as for ce_fwd; rows may be 0.
 * counts       device pointer to two doubles, written: counts[0] = D of
 *              these rows (the count when weight is NULL), counts[1] = the
 *              number of rows that take part (target not ignore_index and in
 *              [0, V); out-of-range targets are reported by ce_fwd).
 * Asynchronous on `stream`; deterministic (fixed-order sums in double).
 * Uses the library scratch of (device, stream), like ce_fwd.
 */
ce_status ce_count(const void* target, const float* weight, int64_t rows, int64_t V,
                   int64_t ignore_index, uint32_t flags, double* counts, ce_stream_t stream);

/*
 * ce_fwd_shard - ce_fwd for one shard of a batch whose counts are known.
 *
 * The caller adds the ce_count outputs of every shard (an all-reduce sum
 * across GPUs, one exchange before the forward) and passes the totals in
 * batch_counts (device pointer to two doubles: D and the number of counted
 * rows of the whole batch). Arguments and outputs are those of ce_fwd,
 * except that the batch totals replace this call's own counts:
 *  - "mean": loss = (sum of this shard's row losses) / D, likewise z_loss,
 *    and the gradient is scaled by 1 / D, so adding the shards' losses gives
 *    the whole batch's mean and every shard's gradient is already the
 *    gradient of that mean;
 *  - "sum" and "mean": acc = (this shard's correct rows) / (the batch's
 *    counted rows), so the shards' values add up to the batch accuracy;
 *  - "none" is unaffected.
 * A shard with no rows writes 0 (not NaN) for loss, z_loss and acc when the
 * batch has counted rows. batch_counts NULL is CE_ERR_INVALID_ARG.
 */
ce_status ce_fwd_shard(void* logits, int dtype, int64_t rows, int64_t V,
                       const void* target, const float* weight, int64_t ignore_index,
                       float label_smoothing, float lse_square_scale, float softcap,
                       int reduction, uint32_t flags, float* loss, float* z_loss,
                       float* acc, int64_t* pred, const double* batch_counts,
                       ce_stream_t stream);

/*
 * ce_fwd_nd - ce_fwd for N-D logits with the class dimension at axis 1,
 * [N, C, d1, ..., dk] (F.cross_entropy's N-D form; tt-mlir pull request
 * #9324, review comments: the reductions run over every non-class
 * dimension). Each position (n, d1..dk) is one row of the ce_fwd
 * definition with V = C, so loss, z_loss, accuracy, predicted tokens and
 * the in-place gradient are those of ce_fwd applied to the logits with the
 * class axis moved last.
 *
 * logits       [N, C, inner] row-major, inner = d1 * ... * dk (inner >= 0;
 *              inner == 1 is exactly ce_fwd with rows = N). Overwritten by
 *              dlogits (same layout) with CE_FLAG_GRAD.
 * target       [N, inner] (int32, or int64 with CE_FLAG_TARGET_I64).
 * loss, z_loss, acc   [N, inner] fp32 for CE_RED_NONE, else [1].
 * pred         [N, inner] int64.
 * Other arguments, results and errors as for ce_fwd. N * inner must stay
 * below 2^31 (CE_ERR_UNSUPPORTED otherwise). For "sum" and "mean" the call
 * enqueues a count kernel before the forward (D and the counted positions
 * land in the library scratch of (device, stream)). Vectorised loads need
 * a 16-byte aligned base and inner a multiple of 16 / sizeof(dtype); other
 * shapes take single-element loads with the same results. Many classes
 * take a form that keeps per-position records in a workspace of (device,
 * stream) that the library allocates on first use and grows when a call
 * needs more (growing frees the old buffer, which waits for the device);
 * a call that must not allocate passes a stream that has already run a
 * call of the same shape.
 */
ce_status ce_fwd_nd(void* logits, int dtype, int64_t N, int64_t C, int64_t inner,
                    const void* target, const float* weight, int64_t ignore_index,
                    float label_smoothing, float lse_square_scale, float softcap,
                    int reduction, uint32_t flags, float* loss, float* z_loss,
                    float* acc, int64_t* pred, ce_stream_t stream);

/*
 * ce_bwd_nd - backward of ce_fwd_nd ("Kernel Profile: CrossEntropy",
 * §Backward Pass): dlogits *= grad_output in place, where grad_output is one
 * fp32 value (grad_per_position == 0) or [N, inner] fp32 values, one per
 * position, multiplying all C classes of that position (reduction "none").
 * A scalar factor of exactly 1.0 leaves dlogits untouched.
 */
ce_status ce_bwd_nd(const float* grad_output, int grad_per_position, void* dlogits,
                    int dtype, int64_t N, int64_t C, int64_t inner, ce_stream_t stream);

/*
 * ce_flce - fused linear cross-entropy: the cross-entropy (as ce_fwd
 * defines it) of the logits hidden @ lm_weight^T + bias, with the gradients
 * of hidden, lm_weight and bias, without materialising more than one chunk
 * of rows of logits ("Kernel Profile: CrossEntropy", closest_existing_kernel:
 * fused_linear_cross_entropy, the cross-entropy kernel extended with the
 * linear layer).
 *
 * hidden       [rows, H] row-major, dtype CE_BF16, CE_F16 or CE_F32.
 * lm_weight    [V, H] row-major, same dtype.
 * bias         [V] fp32, or NULL.
 * target, class_weight, ignore_index, label_smoothing, lse_square_scale,
 * softcap, reduction, flags, loss, z_loss, acc, pred
 *              as for ce_fwd over the [rows, V] logits. With CE_FLAG_GRAD the
 *              gradients of the reduced loss (for "none", of the sum of the
 *              row losses) are written to the non-NULL ones of:
 * grad_hidden  [rows, H] in dtype;
 * grad_weight  [V, H] fp32 (overwritten, not accumulated into);
 * grad_bias    [V] fp32.
 * chunk_rows   rows per chunk (<= 0: about 2 GB of fp32 logits a chunk, a
 *              multiple of 256 rows when at least 256).
 * workspace    device memory of at least ce_flce_workspace_bytes(dtype,
 *              rows, V, chunk_rows) bytes, 256-byte aligned, owned by the
 *              caller; it holds one chunk of fp32 logits (and of the gradient
 *              in dtype) and the chunks' partial sums.
 * Per chunk: logits by this library's tensor-core GEMM (ce_gemm; inputs in
 * dtype, fp32 accumulation), the fused forward of this library in place
 * over them (one shard of the batch, D from ce_count), the gradient rounded
 * to dtype, then grad_hidden = G @ lm_weight and grad_weight += G^T @ hidden
 * (ce_gemm again, fp32 accumulation) and grad_bias += column sums. fp32
 * inputs, and 16-bit ones with H or V not a multiple of 8 or unaligned
 * bases, take cuBLAS for the three GEMMs (GBCE_FLCE_GEMM=cublas forces it).
 * Scalars are added in chunk order: deterministic. Asynchronous on
 * `stream`; uses the library scratch of (device, stream) (and a cuBLAS
 * handle per device on the cuBLAS path).
 * Errors as for ce_fwd; CE_ERR_INVALID_ARG also for a missing or too small
 * workspace.
 */
size_t ce_flce_workspace_bytes(int dtype, int64_t rows, int64_t V, int64_t chunk_rows);

ce_status ce_flce(const void* hidden, const void* lm_weight, const float* bias, int dtype,
                  int64_t rows, int64_t H, int64_t V, const void* target,
                  const float* class_weight, int64_t ignore_index, float label_smoothing,
                  float lse_square_scale, float softcap, int reduction, uint32_t flags,
                  float* loss, float* z_loss, float* acc, int64_t* pred, void* grad_hidden,
                  float* grad_weight, float* grad_bias, int64_t chunk_rows, void* workspace,
                  size_t workspace_bytes, ce_stream_t stream);

/*
 * ce_gemm_abt - C = A @ B^T (+ bias), the logits GEMM of ce_flce, on the
 * tensor cores (tcgen05, operands staged by TMA, fp32 accumulator in tensor
 * memory). A [M, K] and B [N, K] row-major in CE_BF16 or CE_F16 with
 * 16-byte aligned bases and K a multiple of 8 (else CE_ERR_UNSUPPORTED);
 * C [M, N] fp32 row-major, written; bias [N] fp32 or NULL. The method has
 * no counterpart: it is the linear layer the fused linear cross-entropy
 * folds in. A bounded wait that gives up records CE_ERR_TIMEOUT for
 * ce_device_status (that call's C is then invalid).
 */
ce_status ce_gemm_abt(const void* A, const void* B, int dtype, int64_t M, int64_t N,
                      int64_t K, float* C, const float* bias, ce_stream_t stream);

/* What ce_gemm does with the product. */
enum { CE_GEMM_F32 = 0, CE_GEMM_F32_ADD = 1, CE_GEMM_16BIT = 2 };

/*
 * ce_gemm - C = A @ B on the tensor cores, for the three GEMMs of the fused
 * linear cross-entropy (logits = hidden @ lm_weight^T, grad_hidden = G @
 * lm_weight, grad_weight += G^T @ hidden). The method has no counterpart:
 * these are the linear layer the fused linear cross-entropy folds in.
 *
 * A            [M, K] as the math has it, stored K-major (a_mn = 0: row-major
 *              [M, K], K contiguous) or MN-major (a_mn = 1: row-major [K, M],
 *              M contiguous, i.e. the storage of A^T).
 * B            [K, N], stored K-major (b_mn = 0: row-major [N, K]) or MN-major
 *              (b_mn = 1: row-major [K, N]).
 * dtype        CE_BF16 or CE_F16 for both operands; bases 16-byte aligned and
 *              the contiguous dimension a multiple of 8 (K, M or N), else
 *              CE_ERR_UNSUPPORTED.
 * C            [M, N] row-major: fp32 written (c_mode CE_GEMM_F32, plus
 *              bias [N] fp32 when bias is not NULL), fp32 added to
 *              (CE_GEMM_F32_ADD), or rounded to nearest even into dtype
 *              (CE_GEMM_16BIT). bias only with CE_GEMM_F32 (else
 *              CE_ERR_INVALID_ARG).
 * Accumulation in fp32 in tensor memory; K > 0. Asynchronous on `stream`;
 * a bounded wait that gives up records CE_ERR_TIMEOUT for ce_device_status
 * (that call's C is then invalid).
 */
ce_status ce_gemm(const void* A, int a_mn, const void* B, int b_mn, int dtype, int64_t M,
                  int64_t N, int64_t K, void* C, int c_mode, const float* bias,
                  ce_stream_t stream);

/*
 * ce_scale_round - out[i] = in[i] * grad_output[0], rounded to nearest-even
 * into dtype (the backward of ce_flce's fp32 weight gradient for a weight
 * stored in dtype). in [n] fp32, grad_output one fp32 value, out [n] dtype;
 * device pointers; out may equal in only for CE_F32.
 */
ce_status ce_scale_round(const float* in, const float* grad_output, void* out, int dtype,
                         int64_t n, ce_stream_t stream);

/*
 * The unfused form: the four aten ops a decomposed F.cross_entropy graph
 * runs (tt-mlir pull request #9324, the table of decomposed aten ops on
 * [1023, 128256] f32 logits, and the #9339 description: max-shifted
 * log-sum-exp, integer targets with ignore_index, mean/sum/none, zero
 * gradients for an all-ignored batch). Class weights follow the aten
 * operators' definitions. All tensors are [rows, C] row-major device
 * arrays of `dtype` unless stated; fp32 arithmetic; results rounded to
 * nearest-even into the dtype. CE_ERR_INVALID_ARG / CE_ERR_UNSUPPORTED
 * mean nothing was enqueued; out-of-range targets are reported through
 * ce_device_status (CE_ERR_TARGET_RANGE) and those rows are treated as
 * ignored.
 */

/* _log_softmax over the last dimension: out[i, j] = x[i, j] - m_i - log S_i,
 * m_i = max_j x[i, j], S_i = sum_j exp(x[i, j] - m_i). out may equal x. */
ce_status ce_log_softmax(const void* x, void* out, int dtype, int64_t rows, int64_t C,
                         ce_stream_t stream);

/* nll_loss_forward: l_i = -w[t_i] * logp[i, t_i] for rows whose target is
 * not ignore_index (0 otherwise). reduction CE_RED_NONE writes l_i to
 * out[0 .. rows-1] and 0 to total_weight[0]; CE_RED_SUM writes sum l_i to
 * out[0]; CE_RED_MEAN writes sum l_i / W (NaN when W is 0), W = sum of
 * w[t_i] over those rows; both write W to total_weight[0]. out and
 * total_weight are fp32 device pointers; flags may hold CE_FLAG_TARGET_I64.
 * Deterministic (fixed-order double sums). */
ce_status ce_nll_loss_fwd(const void* logp, int dtype, int64_t rows, int64_t C,
                          const void* target, const float* weight, int64_t ignore_index,
                          int reduction, uint32_t flags, float* out, float* total_weight,
                          ce_stream_t stream);

/* nll_loss_backward: writes every element of grad_input: 0, except
 * grad_input[i, t_i] = -w[t_i] * g_i for rows whose target is not
 * ignore_index, g_i = grad_output[i] (CE_RED_NONE), grad_output[0]
 * (CE_RED_SUM) or grad_output[0] / total_weight[0] (CE_RED_MEAN; the
 * forward's total_weight). grad_output and total_weight are fp32 device
 * pointers (total_weight is read for CE_RED_MEAN only). */
ce_status ce_nll_loss_bwd(const float* grad_output, const float* total_weight,
                          void* grad_input, int dtype, int64_t rows, int64_t C,
                          const void* target, const float* weight, int64_t ignore_index,
                          int reduction, uint32_t flags, ce_stream_t stream);

/* _log_softmax_backward_data: grad_input[i, j] = grad_output[i, j]
 * - exp(output[i, j]) * sum_k grad_output[i, k], with output the
 * log-softmax. grad_input may equal grad_output. */
ce_status ce_log_softmax_bwd(const void* grad_output, const void* output, void* grad_input,
                             int dtype, int64_t rows, int64_t C, ce_stream_t stream);

/*
 * ce_bwd - backward (§Backward Pass: the stored gradient times
 * grad_output): dlogits *= grad_output, in place.
 *
 * grad_output  fp32 device pointer: one value (grad_per_row == 0) or one per
 *              row (grad_per_row != 0, for reduction "none").
 * dlogits      [rows, V] in dtype, the buffer ce_fwd wrote with CE_FLAG_GRAD.
 * The kernel reads grad_output on the device; rows whose factor is exactly
 * 1.0 are left untouched, since multiplying by one changes nothing.
 */
ce_status ce_bwd(const float* grad_output, int grad_per_row, void* dlogits,
                 int dtype, int64_t rows, int64_t V, ce_stream_t stream);

/*
 * ce_device_status - synchronizes `stream`, then reads and clears the
 * device-side error word of that stream's scratch area. Returns CE_OK,
 * CE_ERR_TARGET_RANGE, CE_ERR_TIMEOUT or CE_ERR_CUDA.
 *
 * Environment read at each call: GBCE_WAIT_TIMEOUT_MS (default 2000) bounds
 * every device wait of a launch in wall time; GBCE_TEST_STALL_COPY=1 is a
 * test hook that makes CTA 0 of the streaming or register-resident forward
 * kernel leave its first bulk copy out, so that one wait runs out and the
 * call records CE_ERR_TIMEOUT (its outputs are then invalid; nothing
 * faults).
 */
ce_status ce_device_status(ce_stream_t stream);

/* Static text for a status code. */
const char* ce_status_string(ce_status status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* ce_last_error(void);

/*
 * ce_scratch_areas - how many (device, stream) scratch areas ce_fwd and the
 * other allocating calls have made so far in this process (each about
 * 128 KB of device memory, kept until exit). ce_fwd_noalloc and
 * ce_noalloc_status never add one. Not part of the method; a query for
 * callers that budget device memory.
 */
int64_t ce_scratch_areas(void);

#ifdef __cplusplus
}
#endif

#endif /* GBCE_H */
