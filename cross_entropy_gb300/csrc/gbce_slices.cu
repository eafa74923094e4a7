// Combine of vocabulary-slice partials into log-probs (one thread per row).
//
// A vocabulary split across devices leaves each device with the statistics
// of its own columns: the max m_i and sum s_i over its non-target columns,
// and the logits of the targets it holds (vocab_slice_stats).  Once the
// caller has gathered every slice's partials, this merges the (m_i, s_i) in
// slice order -- a fixed order, so the result does not depend on which
// device ran first -- takes each target's logit from the slice that holds
// it, and finishes exactly as the single-device sweep does: the other
// targets join a target's "others", then log p = -softplus(log s + (m -
// x_t) / T).  It also gives each row's whole state -- the max M over all
// its columns and the sum S of exp((x_j - M) / T) -- which the slice
// gradient takes as its exponents' reference for a row whose first index
// lies far below the row's max.
//
// Source: "Fix softmax collapse in CE, GRPO, KL/JSD and softmax"
// (Liger-Kernel PR #1555), "Summary", first bullet (the vocab-parallel form
// reduces both sums; here the caller gathers the partials and this kernel
// reduces them).
#include "gbce_kernels.cuh"

namespace gbce {

__global__ void slice_combine_kernel(const float *partials, int slices, SliceOffsets offs,
                                     int64_t rows, const int64_t *index, int K,
                                     int64_t ignore_index, const uint8_t *row_mask, float T,
                                     float c, float *logp_out, float *target_logit_out,
                                     float *row_state_out, int32_t *dev_status)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= rows)
        return;
    const int64_t vocab = offs.off[slices];
    const int64_t stride = rows * (2 + K);  // one slice's partials
    const int64_t *ix = index + r * K;
    if ((row_mask != nullptr && row_mask[r] == 0) || ix[0] == ignore_index) {
        for (int k = 0; k < K; ++k)
            logp_out[r * K + k] = 0.0f;
        if (target_logit_out)
            target_logit_out[r] = 0.0f;
        if (row_state_out) {
            row_state_out[2 * r] = kNegInf;
            row_state_out[2 * r + 1] = 0.0f;
        }
        return;
    }
    float m = kNegInf, s = 0.0f;
    for (int i = 0; i < slices; ++i) {
        const float *part = partials + i * stride + r * (2 + K);
        merge_max_sum(m, s, part[0], part[1], c);
    }
    int32_t tg[GBCE_MAX_K];
    float xt[GBCE_MAX_K];
    for (int k = 0; k < K; ++k) {
        const int64_t t = ix[k];
        tg[k] = (t >= 0 && t < vocab) ? static_cast<int32_t>(t) : -1;
        xt[k] = 0.0f;
        if (tg[k] >= 0) {
            int owner = 0;
            while (owner + 1 < slices && offs.off[owner + 1] <= t)
                ++owner;
            xt[k] = partials[owner * stride + r * (2 + K) + 2 + k];
        }
    }
    for (int k = 0; k < K; ++k) {
        float out;
        if (tg[k] < 0) {
            out = __int_as_float(0x7fc00000);
            report(dev_status, GBCE_DEV_BAD_INDEX);
        } else {
            out = logp_with_targets<GBCE_MAX_K>(m, s, tg, xt, K, k, c, T);
        }
        logp_out[r * K + k] = out;
    }
    if (target_logit_out)
        target_logit_out[r] = tg[0] >= 0 ? xt[0] : __int_as_float(0x7fc00000);
    if (row_state_out) {
        // the other columns' state with each distinct target folded in
        float M = m, S = s;
        for (int k = 0; k < K; ++k) {
            bool dup = tg[k] < 0;
            for (int i = 0; i < k; ++i)
                dup |= (tg[i] == tg[k]);
            if (!dup)
                merge_max_sum(M, S, xt[k], 1.0f, c);
        }
        row_state_out[2 * r] = M;
        row_state_out[2 * r + 1] = S;
    }
}

cudaError_t launch_slice_combine(const float *partials, int slices, const SliceOffsets &offs,
                                 int64_t rows, const int64_t *index, int64_t k,
                                 int64_t ignore_index, const uint8_t *row_mask, float T, float c,
                                 float *logp_out, float *target_logit_out, float *row_state_out,
                                 int32_t *dev_status, cudaStream_t stream)
{
    if (rows == 0)
        return cudaSuccess;
    const int threads = 128;
    const unsigned blocks = static_cast<unsigned>((rows + threads - 1) / threads);
    slice_combine_kernel<<<blocks, threads, 0, stream>>>(partials, slices, offs, rows, index,
                                                         static_cast<int>(k), ignore_index,
                                                         row_mask, T, c, logp_out,
                                                         target_logit_out, row_state_out,
                                                         dev_status);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace gbce
