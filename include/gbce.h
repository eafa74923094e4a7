/*
 * gbce.h -- C ABI of libgbce.so: row-wise log-softmax and token cross-entropy
 * over a [rows, vocab] logit matrix on one NVIDIA GB300 (sm_103a).
 *
 * What is computed (z_j = x_j / T for a row x of length V, temperature T):
 *
 *   log p_t = -softplus( log sum_{j != t} exp(z_j - m_t) + m_t - z_t ),
 *   m_t     = max_{j != t} z_j,   softplus(a) = max(a,0) + log1p(exp(-|a|)),
 *
 * which equals z_t - logsumexp_j z_j but never rounds to exactly 0 (and is
 * never positive) when the target leads the other logits by a wide margin.
 * This is the collapse-safe form of "Fix softmax collapse in CE, GRPO,
 * KL/JSD and softmax" (Liger-Kernel PR #1555), section "Summary": the first
 * pass also accumulates the sum without the target, and the loss is
 * softplus(log(sum_others) + m - x_y).
 *
 * Conventions shared by every entry point:
 *
 *  - Memory.  Every pointer argument is DEVICE memory owned by the caller,
 *    except that `stream` is a cudaStream_t handle (NULL = legacy default
 *    stream).  The library allocates nothing, frees nothing and keeps no
 *    state between calls; scratch space is the caller's `workspace`.
 *  - Layout.  Logits are row-major: row r starts `r * row_stride` ELEMENTS
 *    after `logits`, and its first `vocab` elements are used.  row_stride >=
 *    vocab.  Index, label, mask and per-row outputs are dense.  The logits
 *    pointer must be aligned to its element size; rows need not be 16-byte
 *    aligned (a misaligned head/tail is read with scalar loads).
 *  - Types.  Logits are fp32 or bf16; every computation is fp32; log-probs,
 *    losses and log-sum-exps are written as fp32; dlogits have the logits'
 *    type (bf16 rounded to nearest even).
 *  - Accuracy.  Against an fp64 evaluation of the same definitions: log-probs,
 *    losses and entropies within 1e-5 to 2e-5 relative; dlogits within 2e-5
 *    (fp32) or 4e-3 (bf16) relative per row.  Confident rows keep these
 *    bounds (the sums run over the non-target columns, the target gradient
 *    is expm1(log p)), down to fp32's subnormals.  A value fp32 cannot hold
 *    at all, such as a log p of -1e-50, is written as 0.  Soft-capped logits
 *    carry the fp32 rounding of cap * tanh(x / cap) in every exponent.  A
 *    backward call takes the forward's fp32 log p and entropy as they are.
 *  - Asynchrony.  Every call only enqueues work on `stream` and returns; it
 *    never synchronizes the host.  The returned status reports HOST-side
 *    argument checks (and launch errors) only.  Some kernels of a call are
 *    programmatic dependents of the kernel before them on the stream (their
 *    launch overlaps it), and each waits for that kernel to complete before
 *    its first global memory access; to the caller a call still runs in
 *    stream order, after all earlier work on `stream` and before all later
 *    work.
 *  - Device-side errors.  A label or index outside [0, vocab) (labels equal
 *    to ignore_index excepted) sets a bit in `*dev_status` (atomic OR; pass
 *    NULL to skip reporting) and makes that row's outputs NaN.  A pipeline
 *    wait that exceeds its time limit sets GBCE_DEV_TIMEOUT and the kernel
 *    returns instead of hanging.  Nothing traps.  The caller zeroes
 *    *dev_status and reads it whenever it likes.
 *  - Threading.  Calls on different streams may run concurrently provided
 *    their output and workspace buffers do not overlap.
 */
#ifndef GBCE_H
#define GBCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GBCE_OK = 0,
    GBCE_EINVAL = 1,     /* null pointer, bad size/stride/temperature, aliasing */
    GBCE_EDTYPE = 2,     /* unsupported dtype or misaligned element pointer */
    GBCE_ECUDA = 3,      /* a CUDA launch or attribute call failed */
    GBCE_EWORKSPACE = 4  /* workspace smaller than gbce_workspace_size() */
} gbce_status;

typedef enum { GBCE_F32 = 0, GBCE_BF16 = 1 } gbce_dtype;

typedef enum { GBCE_NONE = 0, GBCE_SUM = 1, GBCE_MEAN = 2 } gbce_reduction;

/* Bits OR-ed into *dev_status by the kernels. */
#define GBCE_DEV_BAD_LABEL 1   /* a label outside [0, vocab) and != ignore_index */
#define GBCE_DEV_BAD_INDEX 2   /* a gather index outside [0, vocab) */
#define GBCE_DEV_TIMEOUT 4     /* a pipeline wait gave up; outputs of that row are invalid */

/* Largest number of gathered indices per row that selective_logsoftmax takes. */
#define GBCE_MAX_K 16

/*
 * Bytes of workspace that any call on a [rows, vocab] problem with k indices
 * per row needs (k = 1 for the cross-entropy calls).  A pure function of its
 * arguments: no CUDA call, valid for any device.  Returns 0 for rows <= 0.
 */
size_t gbce_workspace_size(int64_t rows, int64_t vocab, int64_t k);

/* Static, human-readable name of a status code. */
const char *gbce_status_string(gbce_status status);

/*
 * Number of kernels this library has enqueued in this process so far (all
 * devices, all streams), for accounting in benchmarks.  Thread-safe.
 */
uint64_t gbce_kernel_launches(void);

/*
 * Selective log-softmax: logp_out[r, k] = log p_{index[r, k]} of row r at
 * temperature T, for rows with row_mask[r] != 0 (or all rows when row_mask
 * is NULL); masked-out rows are not read and get 0.  With entropy_out, the
 * same sweep also gives the entropy of each row's softmax,
 * entropy_out[r] = -sum_j p_j log p_j (0 log 0 = 0; 0 for masked rows),
 * with the dominant column's 1 - p taken from its accurate log p, so a
 * confident row keeps its small positive entropy whichever column it is
 * confident in (when that is not the first index, the row's entropy is
 * recomputed around it in a second pass over that row).
 *
 * Source: "perf(rlhf): chunk selective_log_softmax instead of looping per
 * token" (ms-swift PR #10337), "PR information": the naive
 * gather(logits.log_softmax(-1)) with top-K indices, temperature and a row
 * mask, here in one launch over all rows; accurate log-probs as in "Fix
 * softmax collapse ..." (Liger-Kernel PR #1555), "Summary", second bullet;
 * the entropy taking the others' sum from the same term as the target's
 * log p: the unsloth-zoo #2080 commit quoted there, "Fix", forward bullet.
 *
 *   logits     [rows, row_stride] fp32/bf16
 *   index      [rows, k] int64, 1 <= k <= GBCE_MAX_K; duplicates allowed
 *   row_mask   [rows] uint8 or NULL
 *   logp_out   [rows, k] fp32
 *   entropy_out [rows] fp32 or NULL (NULL: the sweep skips the entropy)
 *   workspace  >= gbce_workspace_size(rows, vocab, k) bytes (may be NULL
 *              when that size is 0), 16-byte aligned
 * Errors: GBCE_EINVAL for NULL logits/index/logp_out with rows > 0,
 * vocab < 1, row_stride < vocab, k outside [1, GBCE_MAX_K], temperature not
 * finite and > 0; GBCE_EDTYPE; GBCE_EWORKSPACE.  Out-of-range indices of
 * live rows: GBCE_DEV_BAD_INDEX and a NaN output for that (r, k); the
 * entropy of a row whose first index is out of range is NaN.
 */
gbce_status selective_logsoftmax(const void *logits, gbce_dtype dtype, int64_t rows,
                                 int64_t vocab, int64_t row_stride, const int64_t *index,
                                 int64_t k, float temperature, const uint8_t *row_mask,
                                 float *logp_out, float *entropy_out, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Selective log-softmax backward: the gradient of sum_k g[r, k] *
 * log p_{index[r, k]} with respect to the logits,
 *   dlogits[r, j] = (1/T) * ( sum_{k : index[r, k] = j} g[r, k] - G_r * p_j ),
 * G_r = sum_k g[r, k], with every gathered column t evaluated as
 *   (1/T) * ( -g_t * expm1(log p_t) - (G_r - g_t) * exp(log p_t) )
 * (g_t = the upstream of every k that gathers t) so that 1 - p_t keeps its
 * value when p_t rounds to 1; masked-out rows get a zero row.  With
 * grad_entropy, the gradient of gH_r * H_r (H_r the row entropy of the
 * forward's entropy_out) is added:
 *   - (gH_r / T) * p_j * (log p_j + H_r)   for every column j,
 * 0 where p_j = 0, with log p of the gathered columns from saved_logp.  The
 * other columns' p_j are taken relative to index[r, 0]; a row with
 * saved_logp[r, 0] < -40 reads its max and sum in a second pass over that
 * row and takes them relative to the max (hundreds of nats between the
 * two would cost fp32 accuracy).
 *
 * Source: the gradient a GRPO-style loss sends back through the accurate
 * log-probs of "Fix softmax collapse in CE, GRPO, KL/JSD and softmax"
 * (Liger-Kernel PR #1555), "Summary", second bullet (-expm1(logp) for
 * 1 - p_y); gradients are part of the checked behaviour of "perf(rlhf):
 * chunk selective_log_softmax instead of looping per token", "PR
 * information".
 *
 *   index       [rows, k] int64, as given to selective_logsoftmax
 *   row_mask    [rows] uint8 or NULL
 *   grad_logp   [rows, k] fp32, device: dL/d logp_out
 *   saved_logp  [rows, k] fp32: selective_logsoftmax's output for the same
 *               logits, index and temperature
 *   grad_entropy  [rows] fp32 or NULL: dL/d entropy_out
 *   saved_entropy [rows] fp32: the forward's entropy_out; NULL exactly when
 *               grad_entropy is NULL
 *   dlogits     [rows, dlogits_row_stride], the logits' dtype; must not
 *               overlap the logits
 * Errors: as ce_bwd; a row with an index outside [0, vocab) sets
 * GBCE_DEV_BAD_INDEX and gets a NaN row.
 */
gbce_status selective_logsoftmax_bwd(const void *logits, gbce_dtype dtype, int64_t rows,
                                     int64_t vocab, int64_t row_stride, const int64_t *index,
                                     int64_t k, float temperature, const uint8_t *row_mask,
                                     const float *grad_logp, const float *saved_logp,
                                     const float *grad_entropy, const float *saved_entropy,
                                     void *dlogits, int64_t dlogits_row_stride,
                                     int32_t *dev_status, void *stream);

/*
 * Options of the token cross-entropy calls (ce_fwd, ce_bwd,
 * ce_fwd_bwd_fused).  A NULL pointer means all defaults (plain CE).
 *
 *   label_smoothing  eps in [0, 1]: the target distribution puts 1 - eps on
 *                    the label and eps / vocab on every class, so a kept
 *                    row's loss is (1 - eps)(-log p_y) + eps * mean_j(-log p_j)
 *                    and its gradient (g/T)(p_j - (1 - eps)[j == y] - eps/vocab),
 *                    the label column in the expm1(log p_y) form ("Fix
 *                    softmax collapse ...", the unsloth-zoo #2080 commit's
 *                    "Fix", backward bullet).  A row with a -inf logit has
 *                    an infinite smoothed loss, as the definition gives.
 *   dft              nonzero: weight each kept row's loss and gradient by its
 *                    own p_y, held constant in the backward (the DFT loss
 *                    -p_y log p_y of ms-swift PR #10353, "PR information").
 *                    Combines with label_smoothing (the weight multiplies
 *                    the smoothed row loss).
 *   softcap          cap >= 0 (0: off): every logit x becomes cap * tanh(x / cap)
 *                    before the temperature and the softmax; the gradient
 *                    with respect to x takes the factor 1 - tanh^2(x / cap).
 *                    Its tanh per element makes these calls ALU-bound, and
 *                    the fused call then runs as a statistics pass and a
 *                    gradient pass.  Logit soft-capping is named among the
 *                    options of the fused losses on "Fix softmax collapse
 *                    ..." (the unsloth-zoo #2080 commit, "Accuracy" tests).
 * ce_bwd must be given the same options as the ce_fwd whose log p it takes.
 * An eps outside [0, 1] (or NaN), or a negative or non-finite softcap, makes
 * the call return GBCE_EINVAL before any GPU work.
 */
typedef struct gbce_ce_options {
    float label_smoothing;
    int32_t dft;
    float softcap;
} gbce_ce_options;

/*
 * Token cross-entropy forward.  For rows whose label is not ignore_index:
 * loss_r = -log p_{labels[r]} at temperature T; ignored rows are skipped
 * before any read of their logits and get loss 0.
 *
 * Source: "Fix softmax collapse ..." (Liger-Kernel PR #1555), "Summary",
 * first bullet (loss = softplus(log(sum_others) + m - x_y)); row selection
 * before any vocabulary work from ms-swift PR #10353, "PR information".
 *
 *   labels      [rows] int64
 *   options     gbce_ce_options or NULL (plain CE)
 *   reduction   GBCE_NONE: loss_out[rows] = loss_r;
 *               GBCE_SUM:  loss_out[0] = sum_r loss_r;
 *               GBCE_MEAN: loss_out[0] = sum_r loss_r / n_items, 0 when
 *               n_items == 0 (all rows ignored).
 *   logp_out    [rows] fp32 or NULL: log p of the label (0 when ignored);
 *               ce_bwd takes it back as saved_logp.
 *   lse_out     [rows] fp32 or NULL: logsumexp_j z_j (0 when ignored).
 *   n_items_out [1] int64 or NULL: number of rows with label != ignore_index.
 *   workspace   >= gbce_workspace_size(rows, vocab, 1) bytes.
 * Sums are deterministic (fixed order) and taken in fp64.
 * Errors: as selective_logsoftmax; bad labels set GBCE_DEV_BAD_LABEL and
 * give NaN for that row (and hence a NaN sum/mean).
 */
gbce_status ce_fwd(const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab,
                   int64_t row_stride, const int64_t *labels, int64_t ignore_index,
                   float temperature, gbce_reduction reduction,
                   const gbce_ce_options *options, float *loss_out,
                   float *logp_out, float *lse_out, int64_t *n_items_out, void *workspace,
                   size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Token cross-entropy backward from saved statistics:
 *   dlogits[r, j] = (g_r / T) * exp(z_j - z_y + log p_y)   for j != y,
 *   dlogits[r, y] = (g_r / T) * expm1(log p_y),
 * i.e. g_r * (softmax - onehot) / T with the target term in the form that
 * does not round to zero (with options: the smoothed and DFT-weighted
 * gradient described at gbce_ce_options); ignored rows get a zero row.  A
 * row with log p_y < -40 evaluates its exponents from the row's max instead
 * (z_j - z_max - log S), read in a second pass over that row: taken
 * relative to the label, a column hundreds of nats above it would lose fp32
 * accuracy.  g_r = grad_out[r]
 * (NONE), grad_out[0] (SUM) or grad_out[0] / n_items (MEAN, 0 when
 * n_items == 0).
 *
 * Source: ms-swift PR #10353, "PR information", second bullet (backward
 * computed directly as g*softmax - g*onehot, zero weight for ignored
 * labels, a separate gradient buffer); the target term -expm1(log p_t) from
 * the unsloth-zoo #2080 commit quoted on "Fix softmax collapse ..."
 * (section "Fix", backward bullet).
 *
 *   grad_out    [rows] (NONE) or [1] fp32, device
 *   saved_logp  [rows] fp32 from ce_fwd's logp_out (same logits, labels, T)
 *   n_items     [1] int64 from ce_fwd; required for GBCE_MEAN, else ignored
 *   dlogits     [rows, dlogits_row_stride] of the logits' dtype; must not
 *               overlap the logits; dlogits_row_stride >= vocab
 * Errors: GBCE_EINVAL for NULL required pointers, overlap, bad strides or
 * temperature; bad labels set GBCE_DEV_BAD_LABEL and give a NaN row.
 */
gbce_status ce_bwd(const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab,
                   int64_t row_stride, const int64_t *labels, int64_t ignore_index,
                   float temperature, gbce_reduction reduction,
                   const gbce_ce_options *options, const float *grad_out,
                   const float *saved_logp, const int64_t *n_items, void *dlogits,
                   int64_t dlogits_row_stride, int32_t *dev_status, void *stream);

/*
 * Cross-entropy forward and backward in one call: the outputs of ce_fwd
 * and, with the upstream gradient known in advance, those of ce_bwd.  Each
 * row's logits are read from HBM once; the gradient pass re-reads them from
 * on-chip memory or L2.
 *
 * Source: as ce_fwd and ce_bwd; taking the gradient in the forward when the
 * upstream gradient is known follows the fused losses described in the
 * unsloth-zoo #2079 commit on "Fix softmax collapse ..." ("Summary").
 *
 * Arguments as in ce_fwd and ce_bwd; loss_out, dlogits and grad_out are
 * required, logp_out / lse_out / n_items_out are optional.
 */
gbce_status ce_fwd_bwd_fused(const void *logits, gbce_dtype dtype, int64_t rows,
                             int64_t vocab, int64_t row_stride, const int64_t *labels,
                             int64_t ignore_index, float temperature,
                             gbce_reduction reduction, const gbce_ce_options *options,
                             const float *grad_out, float *loss_out,
                             float *logp_out, float *lse_out, int64_t *n_items_out,
                             void *dlogits, int64_t dlogits_row_stride, void *workspace,
                             size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Vocabulary-parallel selective log-softmax: the vocabulary is split into
 * slices (e.g. one per device, as a vocab-parallel LM head leaves it), each
 * slice's statistics are computed where its logits are, the caller gathers
 * them (any transport: an all-gather over devices, or nothing when every
 * slice is on one device), and one combine gives the log-probs.  The
 * gradient is then computed slice by slice from the combined log-probs.
 * Token cross-entropy is the case k = 1, index = labels, ignore_index = the
 * ignored label: loss_r = -logp[r], and its gradient is vocab_slice_grad
 * with grad_logp[r] = -(upstream of row r).
 *
 * Source: "Fix softmax collapse in CE, GRPO, KL/JSD and softmax"
 * (Liger-Kernel PR #1555), "Summary", first bullet: the vocab-parallel form
 * keeps, per slice, the sum over the columns other than the target, and
 * reduces both sums across slices.
 *
 * Slices are described by their global column ranges: slice i holds columns
 * [slice_offsets[i], slice_offsets[i + 1]) of a vocabulary of `vocab`
 * columns, slice_offsets[0] = 0 and slice_offsets[slices] = vocab.
 * Indices are global columns.  A row is skipped (log p 0, zero gradient)
 * when row_mask[r] == 0 or index[r, 0] == ignore_index.  Label smoothing,
 * DFT, soft-capping and the entropy are not available on this path.
 */
#define GBCE_MAX_SLICES 64

/*
 * Statistics of one slice.  logits: [rows, row_stride] holding the slice's
 * slice_vocab columns, global columns [vocab_offset, vocab_offset +
 * slice_vocab).  partials: [rows, 2 + k] fp32, device, written as
 *   partials[r, 0] = m_r = max over the slice's non-target columns of x / T
 *                    (in units of x, i.e. the raw max),
 *   partials[r, 1] = sum of exp((x_j - m_r) / T) over those columns,
 *   partials[r, 2 + k'] = logit of index[r, k'] if this slice holds it, else 0;
 * a skipped row gets (-inf, 0, 0, ...).
 * Errors: as selective_logsoftmax; GBCE_EINVAL also for vocab_offset < 0 or
 * vocab_offset + slice_vocab > vocab.  Indices outside [0, vocab) are
 * reported by the combine.
 */
gbce_status vocab_slice_stats(const void *logits, gbce_dtype dtype, int64_t rows,
                              int64_t slice_vocab, int64_t row_stride, int64_t vocab_offset,
                              int64_t vocab, const int64_t *index, int64_t k,
                              int64_t ignore_index, const uint8_t *row_mask, float temperature,
                              float *partials, int32_t *dev_status, void *stream);

/*
 * Combine of all slices' partials, stacked in slice order as
 * partials[slices, rows, 2 + k] (device).  slice_offsets: HOST array of
 * slices + 1 int64 (read during the call).  logp_out: [rows, k] fp32 as
 * selective_logsoftmax would give on the whole vocabulary (a bad index: NaN
 * and GBCE_DEV_BAD_INDEX); target_logit_out: [rows] fp32 or NULL, the logit
 * of index[r, 0], which vocab_slice_grad needs; row_state_out: [rows, 2]
 * fp32 or NULL, each row's max M over all its columns (raw logit) and S =
 * sum_j exp((x_j - M) / T) (a skipped row: -inf, 0), which vocab_slice_grad
 * takes for rows far below their max.  The merge runs in slice
 * order, so the result does not depend on the order the slices were
 * computed in.
 * Errors: GBCE_EINVAL for slices outside [1, GBCE_MAX_SLICES], offsets not
 * starting at 0 or not increasing, k outside [1, GBCE_MAX_K], a bad
 * temperature or NULL required pointers.
 */
gbce_status vocab_slice_combine(const float *partials, int64_t slices,
                                const int64_t *slice_offsets, int64_t rows, const int64_t *index,
                                int64_t k, int64_t ignore_index, const uint8_t *row_mask,
                                float temperature, float *logp_out, float *target_logit_out,
                                float *row_state_out, int32_t *dev_status, void *stream);

/*
 * Gradient of sum_k grad_logp[r, k] * logp[r, k] with respect to one
 * slice's logits (the columns of selective_logsoftmax_bwd that the slice
 * holds), from the combined log-probs and target logit:
 *   dlogits[r, j] = (1/T) (sum_{k : index[r, k] = j} g[r, k] - G_r p_j),
 *   p_j = exp((x_j - x_{t0}) / T + logp[r, 0]),
 * gathered columns in the -expm1 form.  A row with logp[r, 0] < -40 and a
 * row_state takes p_j = exp((x_j - M) / T) / S from the row state instead:
 * taken relative to index 0, a column hundreds of nats above it would lose
 * fp32 accuracy.
 *   logp         [rows, k] fp32 from vocab_slice_combine
 *   target_logit [rows] fp32 from vocab_slice_combine
 *   row_state    [rows, 2] fp32 from vocab_slice_combine, or NULL
 *   dlogits      [rows, dlogits_row_stride] of the logits' type, the slice's
 *                columns; must not overlap the logits
 * Errors: as selective_logsoftmax_bwd; a row with an index outside
 * [0, vocab) gets a NaN row and GBCE_DEV_BAD_INDEX.
 */
gbce_status vocab_slice_grad(const void *logits, gbce_dtype dtype, int64_t rows,
                             int64_t slice_vocab, int64_t row_stride, int64_t vocab_offset,
                             int64_t vocab, const int64_t *index, int64_t k, int64_t ignore_index,
                             const uint8_t *row_mask, float temperature, const float *grad_logp,
                             const float *logp, const float *target_logit,
                             const float *row_state, void *dlogits, int64_t dlogits_row_stride,
                             int32_t *dev_status, void *stream);

/*
 * ce_fwd_bwd_fused without a caller workspace and without any allocation.
 *
 * The pages have no counterpart: this exists for callers that cannot provide
 * scratch memory -- a C program or plugin without a device allocator of its
 * own, which must not call cudaMalloc on its hot path (cudaMalloc can
 * synchronize the device, and next to a framework's caching allocator it can
 * fail or fragment memory).  The scratch is a fixed array of
 * GBCE_NOALLOC_SCRATCH_BYTES bytes inside the library's device image, held on
 * every GPU that loads the library until the process exits.
 *
 * Arguments and results are those of ce_fwd_bwd_fused minus the workspace.
 * Returns GBCE_EWORKSPACE, before any GPU work, when
 * gbce_workspace_size(rows, vocab, 1) > GBCE_NOALLOC_SCRATCH_BYTES (about
 * 130 000 rows).  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and keeps it for
 * the rest of the process; make that first call before any stream capture.
 * The kept address belongs to the device's primary context as it was then:
 * after cudaDeviceReset (or any other reset of that context) it is stale,
 * so a program that resets a device must not call this entry point on it
 * afterwards.  All calls share the one array: calls whose GPU work overlaps
 * (e.g. on two streams) race and must be serialized by the caller.  Nothing
 * in the array needs zeroing beforehand: each call writes every scratch
 * value it reads (the item count, the row ticket, the per-row losses) first.
 */
#define GBCE_NOALLOC_SCRATCH_BYTES (1u << 20)
gbce_status ce_fwd_bwd_fused_noalloc(const void *logits, gbce_dtype dtype, int64_t rows,
                                     int64_t vocab, int64_t row_stride, const int64_t *labels,
                                     int64_t ignore_index, float temperature,
                                     gbce_reduction reduction, const float *grad_out,
                                     float *loss_out, float *logp_out, float *lse_out,
                                     int64_t *n_items_out, void *dlogits,
                                     int64_t dlogits_row_stride, int32_t *dev_status,
                                     void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GBCE_H */
