// Item count and loss reduction over rows (one CTA each).
//
// n_items = number of rows whose label is not ignore_index, counted exactly
// in int64; the reduced loss is sum_r loss_r (SUM) or that sum / n_items
// (MEAN, 0 when every row is ignored).  Every thread sums a fixed strided
// subset of rows in order and the partials are combined in a fixed tree, so
// the result is bit-identical from run to run.  Accumulation is fp64: it
// touches rows values, not rows x vocab, so its cost is negligible.
//
// Source: the per-token losses scattered back and reduced over supervised
// tokens, ms-swift PR #10353, "PR information"; mean over num_items as in
// the unsloth-zoo #2079 commit ("batchmean or num_items_in_batch").
#include "gbce_device.cuh"
#include "gbce_internal.h"

namespace gbce {

constexpr int kReduceThreads = 1024;

__device__ int64_t block_sum_i64(int64_t v, int64_t *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (kReduceThreads / 32) ? scratch[lane] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, off);
    }
    __syncthreads();
    return v;  // valid in thread 0
}

__device__ double block_sum_f64(double v, double *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0)
        scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (kReduceThreads / 32) ? scratch[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, off);
    }
    __syncthreads();
    return v;  // valid in thread 0
}

__device__ int64_t count_items(const int64_t *labels, int64_t rows, int64_t ignore_index,
                               int64_t *scratch)
{
    int64_t n = 0;
    int64_t r0 = 0;
    if ((reinterpret_cast<uintptr_t>(labels) & 15u) == 0) {
        // two labels per 16-byte load, several loads in flight per thread
        const longlong2 *v = reinterpret_cast<const longlong2 *>(labels);
        const int64_t nv = rows / 2;
#pragma unroll 4
        for (int64_t i = threadIdx.x; i < nv; i += kReduceThreads) {
            const longlong2 w = v[i];
            n += (w.x != ignore_index) + (w.y != ignore_index);
        }
        r0 = nv * 2;
    }
    for (int64_t r = r0 + threadIdx.x; r < rows; r += kReduceThreads)
        n += (labels[r] != ignore_index);
    return block_sum_i64(n, scratch);
}

__global__ void __launch_bounds__(kReduceThreads)
    count_items_kernel(const int64_t *labels, int64_t rows, int64_t ignore_index, int64_t *n_out,
                       int32_t *zero_out)
{
    __shared__ int64_t scratch[kReduceThreads / 32];
    if (threadIdx.x == 0 && zero_out != nullptr)
        *zero_out = 0;
    const int64_t n = count_items(labels, rows, ignore_index, scratch);
    if (threadIdx.x == 0)
        *n_out = n;
}

__global__ void __launch_bounds__(kReduceThreads)
    reduce_loss_kernel(const float *loss_rows, const int64_t *labels, int64_t rows,
                       int64_t ignore_index, int reduction, const int64_t *n_in,
                       int64_t *count_into, float *loss_out)
{
    __shared__ int64_t iscratch[kReduceThreads / 32];
    __shared__ double dscratch[kReduceThreads / 32];
    __shared__ int64_t s_n;
    if (count_into != nullptr) {
        const int64_t n = count_items(labels, rows, ignore_index, iscratch);
        if (threadIdx.x == 0) {
            *count_into = n;
            s_n = n;
        }
    } else if (threadIdx.x == 0) {
        s_n = n_in != nullptr ? *n_in : 0;
    }
    // per-thread partial over a fixed set of rows, in a fixed order
    double acc = 0.0;
    int64_t r0 = 0;
    if ((reinterpret_cast<uintptr_t>(loss_rows) & 15u) == 0) {
        const float4 *v = reinterpret_cast<const float4 *>(loss_rows);
        const int64_t nv = rows / 4;
#pragma unroll 4
        for (int64_t i = threadIdx.x; i < nv; i += kReduceThreads) {
            const float4 w = v[i];
            acc += (static_cast<double>(w.x) + static_cast<double>(w.y)) +
                   (static_cast<double>(w.z) + static_cast<double>(w.w));
        }
        r0 = nv * 4;
    }
    for (int64_t r = r0 + threadIdx.x; r < rows; r += kReduceThreads)
        acc += static_cast<double>(loss_rows[r]);
    const double total = block_sum_f64(acc, dscratch);  // ends with __syncthreads
    if (threadIdx.x == 0) {
        double out = total;
        if (reduction == 2)
            out = s_n > 0 ? total / static_cast<double>(s_n) : 0.0;
        *loss_out = static_cast<float>(out);
    }
}

cudaError_t launch_count_items(const int64_t *labels, int64_t rows, int64_t ignore_index,
                               int64_t *n_out, int32_t *zero_out, cudaStream_t stream)
{
    count_items_kernel<<<1, kReduceThreads, 0, stream>>>(labels, rows, ignore_index, n_out,
                                                         zero_out);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_reduce_loss(const float *loss_rows, const int64_t *labels, int64_t rows,
                               int64_t ignore_index, int reduction, const int64_t *n_in,
                               int64_t *count_into, float *loss_out, cudaStream_t stream)
{
    reduce_loss_kernel<<<1, kReduceThreads, 0, stream>>>(loss_rows, labels, rows, ignore_index,
                                                         reduction, n_in, count_into, loss_out);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace gbce
