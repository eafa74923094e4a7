// Which row kernel runs a launch (included by the per-type translation units).
#pragma once

#include "gbce_persistent.cuh"

namespace gbce {

// Rows of a fused call are split across a cluster of C CTAs so that each
// CTA's slice is at most kFusedSliceBytes: the slice is what must stay in L2
// between the statistics pass and the gradient pass, and 2 CTAs per SM x
// 152 SMs x 80 KB = 24 MB stays well inside the 126 MB L2 next to the
// dlogits stream.  C is at most the portable cluster size of 8.
constexpr int64_t kFusedSliceBytes = 80 * 1024;

template <typename T>
int fused_cluster_size(int64_t vocab)
{
    const int64_t bytes = vocab * static_cast<int64_t>(sizeof(T));
    const int64_t C = (bytes + kFusedSliceBytes - 1) / kFusedSliceBytes;
    return static_cast<int>(C < 1 ? 1 : (C > kMaxClusterCtas ? kMaxClusterCtas : C));
}

// Kernel choice for a row launch: a fused cross-entropy call over many rows
// runs the persistent kernel (one CTA per SM walking rows); build options
// select instead a cluster of CTAs per row (partials swapped through
// distributed shared memory) or one CTA per row.  Everything else runs one
// CTA per (row, vocab slice).
template <typename T>
cudaError_t launch_rows_dispatch(const RowParams &p, int mode, cudaStream_t stream)
{
    if (mode == kModeFused && p.splits == 1 && p.ls_eps != 0.0f) {
        // label smoothing needs each row's sum of logits, which only the
        // persistent kernel carries among the fused designs
        const int sms = device_sm_count();
        if (sms <= 0)
            return cudaErrorInvalidDevice;
        return launch_persistent_fused<T>(p, static_cast<int>(p.rows < sms ? p.rows : sms), stream);
    }
    if (mode == kModeFused && p.splits == 1) {
#if defined(GBCE_FUSED_CLUSTER)  // build option: a cluster of CTAs per row
        const int C = fused_cluster_size<T>(p.vocab);
        if (C > 1 && p.rows * C <= INT32_MAX) {
            RowParams q = p;
            q.splits = C;
            return launch_fused_row_cluster<T>(q, stream);
        }
#elif !defined(GBCE_FUSED_PER_ROW)  // build option: one CTA per row
        const int sms = device_sm_count();
        if (sms > 0)
            return launch_persistent_fused<T>(p, static_cast<int>(p.rows < sms ? p.rows : sms),
                                              stream);
#endif
    }
    return launch_rows_per_unit<T>(p, mode, stream);
}

}  // namespace gbce
