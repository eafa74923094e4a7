// ce_fwd_bwd_fused_noalloc: the fused cross-entropy call for callers that
// cannot hand the library a workspace.
//
// Who needs it: a plain C program or a plugin loaded into someone else's
// process often has no device allocator to draw a workspace from, and must
// not call cudaMalloc on its hot path -- cudaMalloc can synchronize the whole
// device (stalling every stream) and, next to a framework's caching
// allocator that already holds most of the memory, it can fail or fragment.
// This entry point needs no workspace from the caller and allocates nothing
// itself: its scratch is one fixed array in the library's device image.
//
// Scratch: `g_noalloc_scratch`, GBCE_NOALLOC_SCRATCH_BYTES bytes, a file-scope
// __device__ array.  Every GPU that loads libgbce.so keeps it until the
// process exits.  Host code cannot use the array's name as a device address,
// so on the first call on each device (with that device current) we ask the
// runtime for its address with cudaGetSymbolAddress and cache it per device.
//
// The array is shared by all calls and keeps whatever the last call left in
// it.  Nothing in it has to start at zero: the fused call writes every part
// of its workspace it reads (item count, the persistent kernel's row ticket
// and row order, per-row losses, per-row log p) before reading it.  Two calls whose GPU
// work overlaps in time (for example on two streams) use the same array and
// race; serialize them.  The looked-up address is kept for the process: it
// goes stale if the device's primary context is reset (cudaDeviceReset).
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gbce.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[GBCE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxCachedDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxCachedDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device.  Returns nullptr if the runtime cannot provide it.
void *scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (dev >= 0 && dev < kMaxCachedDevices && g_scratch_ptr[dev] != nullptr)
        return g_scratch_ptr[dev];
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess)
        return nullptr;
    if (dev >= 0 && dev < kMaxCachedDevices)
        g_scratch_ptr[dev] = ptr;
    return ptr;
}

}  // namespace

extern "C" gbce_status ce_fwd_bwd_fused_noalloc(
    const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab, int64_t row_stride,
    const int64_t *labels, int64_t ignore_index, float temperature, gbce_reduction reduction,
    const float *grad_out, float *loss_out, float *logp_out, float *lse_out,
    int64_t *n_items_out, void *dlogits, int64_t dlogits_row_stride, int32_t *dev_status,
    void *stream)
{
    // Refuse problems whose scratch would not fit before touching the GPU.
    if (rows < 0 || vocab < 1)
        return GBCE_EINVAL;
    if (gbce_workspace_size(rows, vocab, 1) > GBCE_NOALLOC_SCRATCH_BYTES)
        return GBCE_EWORKSPACE;
    void *scratch = nullptr;
    if (rows > 0) {
        scratch = scratch_on_current_device();
        if (scratch == nullptr)
            return GBCE_ECUDA;
    }
    return ce_fwd_bwd_fused(logits, dtype, rows, vocab, row_stride, labels, ignore_index,
                            temperature, reduction, nullptr, grad_out, loss_out, logp_out, lse_out,
                            n_items_out, dlogits, dlogits_row_stride, scratch,
                            GBCE_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
