// Internal interface between the C-ABI layer (gbce_api.cu) and the kernel
// translation units (one per logit type).  Not installed, not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbce {

// Counts every kernel the library enqueues (see gbce_kernel_launches()).
void note_launches(int n);

// Streaming multiprocessors of the current device (cached per device; 0 if
// the runtime cannot say).
int device_sm_count();

// What a row-kernel launch does with each (row, vocab slice) work unit.
enum Mode : int {
    kModeLogp = 0,   // selective log-softmax statistics (K gathered indices)
    kModeCe = 1,     // cross-entropy forward statistics (label, ignore_index)
    kModeGrad = 2,   // cross-entropy gradient from saved log p (ce_bwd)
    kModeFused = 3,  // statistics then gradient of the same row (one launch)
    kModeLogpGrad = 4,  // selective log-softmax gradient from saved log p (K indices)
    kModeLogpEnt = 5,   // kModeLogp plus the entropy of each row
    kModeLogpEntGrad = 6,  // kModeLogpGrad plus the gradient of the row entropy
    kModeCeSmooth = 7,     // kModeCe plus the sum of each row's logits (label smoothing)
    kModeCeCap = 8,        // kModeCe on soft-capped logits cap * tanh(x / cap)
    kModeGradCap = 9,      // kModeGrad on soft-capped logits, with the chain factor
    kModeCeCapSmooth = 10,  // kModeCeCap plus the sum of each row's capped logits
    kModeSliceStats = 11,   // a vocabulary slice's (max, sum) and target logits (partials)
};

struct RowParams {
    const void *logits;
    int64_t rows, vocab, row_stride;  // row_stride in elements

    const int64_t *targets;  // kModeLogp: index [rows, k]; otherwise labels [rows]
    int64_t k;               // gathered indices per row (1 for the CE modes)
    int64_t ignore_index;
    const uint8_t *row_mask;  // kModeLogp, nullable

    float T;  // temperature
    float c;  // log2(e) / T
    float ls_eps;  // CE label smoothing (0: none)
    int dft;       // CE: weight each row's loss and gradient by its detached p_y
    float softcap, inv_cap;  // CE logit soft-capping (kModeCeCap / kModeGradCap)
    int splits;  // vocab slices per row: 1, or the CTAs of a row's cluster (<= 8)

    float *logp_out;   // kModeLogp: [rows, k]; CE modes: [rows] or null
    float *loss_rows;  // CE modes: [rows]
    float *lse_out;    // CE modes: [rows] or null
    float *entropy_out;  // kModeLogpEnt: [rows]

    void *dlogits;  // kModeGrad / kModeFused
    int64_t d_stride;
    int vec_store;  // dlogits rows share the logits rows' 16-byte phase
    const float *grad_out;    // CE: [rows] or [1]; kModeLogpGrad: [rows, k]
    int reduction;  // 0 none, 1 sum, 2 mean
    const int64_t *n_items;
    const float *saved_logp;  // kModeGrad: [rows]; kModeLogpGrad: [rows, k]
    const float *grad_entropy;   // kModeLogpEntGrad: [rows] dL/dH
    const float *saved_entropy;  // kModeLogpEntGrad: [rows] H from the forward

    int32_t *dev_status;
    int32_t *row_ticket;  // persistent fused kernel: rows handed out beyond the first wave
    // persistent fused kernel: the order rows are handed out in (live rows
    // first, then ignored ones), valid when *row_order_flag != 0; nullable
    const int32_t *row_order;
    const int32_t *row_order_flag;
    // one-CTA-per-row launches of more than one wave: each CTA warms in L2
    // the start of the row this many rows ahead (about the CTA that takes
    // its place on the SM); 0 for none
    int64_t prefetch_ahead;

    // Vocabulary-slice calls (vocab_total > 0): the logits hold global
    // columns [vocab_offset, vocab_offset + vocab); targets are global
    // indices in [0, vocab_total); rows whose first index equals
    // ignore_index are skipped like masked rows.
    int64_t vocab_offset, vocab_total;
    float *slice_partials;      // kModeSliceStats: [rows, 2 + k] (m, s, target logits)
    const float *target_logit;  // slice gradient: [rows] logit of the first index
    // slice gradient: [rows, 2] the whole row's max M (raw logit) and sum S of
    // 2^{(x_j - M) c} over all its columns, from the combine; nullable
    const float *row_state;
};

// Merge vocabulary-slice partials into log-probs (one thread per row).
struct SliceOffsets {
    static constexpr int kMax = 64;
    int64_t off[kMax + 1];
};
cudaError_t launch_slice_combine(const float *partials, int slices, const SliceOffsets &offs,
                                 int64_t rows, const int64_t *index, int64_t k,
                                 int64_t ignore_index, const uint8_t *row_mask, float T, float c,
                                 float *logp_out, float *target_logit_out, float *row_state_out,
                                 int32_t *dev_status,
                                 cudaStream_t stream);

// Row kernel (one CTA per work unit) for logit type T (float / bf16).
template <typename T>
cudaError_t launch_rows(const RowParams &p, int mode, cudaStream_t stream);

// n_items = #(labels != ignore_index) into *n_out (one CTA); also zeroes
// *zero_out when it is non-null (the persistent kernel's row ticket).
// n_items of the labels; zero_out (nullable) is zeroed; with order_out
// (nullable, [rows]) the rows are also listed live first, then ignored, each
// group in row order, when most rows are ignored, and *order_flag says
// whether that order was written (0: the identity order).
cudaError_t launch_count_items(const int64_t *labels, int64_t rows, int64_t ignore_index,
                               int64_t *n_out, int32_t *zero_out, int32_t *order_out,
                               int32_t *order_flag, cudaStream_t stream);

// loss_out[0] = sum (SUM) or sum / n (MEAN, 0 when n == 0) of loss_rows in a
// fixed order with fp64 accumulation; when count_into is non-null the item
// count is computed first and stored there (and used for MEAN).
cudaError_t launch_reduce_loss(const float *loss_rows, const int64_t *labels, int64_t rows,
                               int64_t ignore_index, int reduction, const int64_t *n_in,
                               int64_t *count_into, float *loss_out, cudaStream_t stream);

}  // namespace gbce
