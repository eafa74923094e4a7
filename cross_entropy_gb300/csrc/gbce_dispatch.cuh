// Which kernel runs a row launch (included by the per-type translation units).
#pragma once

#include "gbce_persistent.cuh"

namespace gbce {

// A fused cross-entropy call over many rows (no vocabulary split) runs the
// persistent kernel: one CTA per SM (two for the soft-capped one) walking
// rows, each row's gradient pass re-reading it from L2.  Everything else
// runs one CTA per (row, vocab slice), the slices of a split row as one
// thread-block cluster.
template <typename T>
cudaError_t launch_rows_dispatch(const RowParams &p, int mode, cudaStream_t stream)
{
    if (mode == kModeFused && p.splits == 1) {
        const int sms = device_sm_count();
        if (sms <= 0)
            return cudaErrorInvalidDevice;
        return launch_persistent_fused<T>(p, sms, stream);
    }
    return launch_rows_per_unit<T>(p, mode, stream);
}

}  // namespace gbce
