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

// One CTA of 256 threads: the inputs are a few rows' worth of bytes, so the
// time is latency -- both arrays are read in one loop (their loads in flight
// together) and both sums go through one block reduction.
constexpr int kReduceThreads = 256;
constexpr int kReduceWarps = kReduceThreads / 32;

// Block-wide sums of an int64 and an fp64 in a fixed tree; valid in thread 0.
__device__ void block_sum2(int64_t &n, double &s, int64_t *iscratch, double *dscratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        n += __shfl_xor_sync(0xffffffffu, n, off);
        s += __shfl_xor_sync(0xffffffffu, s, off);
    }
    if (lane == 0) {
        iscratch[warp] = n;
        dscratch[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
        n = lane < kReduceWarps ? iscratch[lane] : 0;
        s = lane < kReduceWarps ? dscratch[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            n += __shfl_xor_sync(0xffffffffu, n, off);
            s += __shfl_xor_sync(0xffffffffu, s, off);
        }
    }
}

// This thread's count of rows with label != ignore_index and (when loss_rows
// is non-null) its fp64 sum of their losses, over a fixed strided subset of
// rows in a fixed order; four rows per step when both arrays are 16-byte
// aligned.
__device__ void thread_partials(const float *loss_rows, const int64_t *labels, int64_t rows,
                                int64_t ignore_index, bool count, int64_t &n, double &s)
{
    n = 0;
    s = 0.0;
    int64_t r0 = 0;
    const bool lab_vec = !count || (reinterpret_cast<uintptr_t>(labels) & 15u) == 0;
    const bool loss_vec = loss_rows == nullptr || (reinterpret_cast<uintptr_t>(loss_rows) & 15u) == 0;
    if (lab_vec && loss_vec) {
        const int64_t nv = rows / 4;
#pragma unroll 2
        for (int64_t i = threadIdx.x; i < nv; i += kReduceThreads) {
            if (count) {
                const longlong2 a = reinterpret_cast<const longlong2 *>(labels)[2 * i];
                const longlong2 b = reinterpret_cast<const longlong2 *>(labels)[2 * i + 1];
                n += (a.x != ignore_index) + (a.y != ignore_index) + (b.x != ignore_index) +
                     (b.y != ignore_index);
            }
            if (loss_rows != nullptr) {
                const float4 w = reinterpret_cast<const float4 *>(loss_rows)[i];
                s += (static_cast<double>(w.x) + static_cast<double>(w.y)) +
                     (static_cast<double>(w.z) + static_cast<double>(w.w));
            }
        }
        r0 = nv * 4;
    }
    for (int64_t r = r0 + threadIdx.x; r < rows; r += kReduceThreads) {
        if (count)
            n += (labels[r] != ignore_index);
        if (loss_rows != nullptr)
            s += static_cast<double>(loss_rows[r]);
    }
}

// The count, and for the persistent fused kernel the order it hands rows
// out in: live rows first, then the ignored ones (each group in row order),
// so that the cheap ignored rows, which only write zeros, come last and
// even out the CTAs' finishing times.  Written only when most rows are
// ignored (sparse supervision: 0.494 -> 0.478 ms at 8192 rows, 25%
// labelled); with a few ignored rows spread among the others it costs time
// instead (2048 rows, 10% ignored: 0.207 -> 0.209 ms), as their zero writes
// then bunch up at the end rather than mixing with the other rows' reads.
// A stable partition, 256 rows at a time, by warp ballots and a scan over
// the eight warps.
__global__ void __launch_bounds__(kReduceThreads)
    count_items_kernel(const int64_t *labels, int64_t rows, int64_t ignore_index, int64_t *n_out,
                       int32_t *zero_out, int32_t *order_out, int32_t *order_flag)
{
    __shared__ int64_t iscratch[kReduceWarps];
    __shared__ double dscratch[kReduceWarps];
    __shared__ int64_t s_live;
    __shared__ int32_t s_wl[kReduceWarps], s_wi[kReduceWarps];
    // the row kernel after this one may start its prologue now: it waits
    // for this kernel's outputs before it reads them
    launch_dependents();
    if (threadIdx.x == 0 && zero_out != nullptr)
        *zero_out = 0;
    int64_t n;
    double s;
    thread_partials(nullptr, labels, rows, ignore_index, true, n, s);
    block_sum2(n, s, iscratch, dscratch);
    if (threadIdx.x == 0) {
        *n_out = n;
        s_live = n;
        if (order_flag != nullptr)
            *order_flag = (order_out != nullptr && 2 * n < rows) ? 1 : 0;
    }
    __syncthreads();
    const int64_t live = s_live;
    if (order_out == nullptr || order_flag == nullptr || 2 * live >= rows)
        return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned below = (1u << lane) - 1u;
    int64_t base_live = 0, base_ign = live;
    for (int64_t t0 = 0; t0 < rows; t0 += kReduceThreads) {
        const int64_t r = t0 + threadIdx.x;
        const bool in = r < rows;
        const bool is_live = in && labels[r] != ignore_index;
        const unsigned bl = __ballot_sync(0xffffffffu, is_live);
        const unsigned bi = __ballot_sync(0xffffffffu, in && !is_live);
        if (lane == 0) {
            s_wl[warp] = __popc(bl);
            s_wi[warp] = __popc(bi);
        }
        __syncthreads();
        int32_t off_l = 0, off_i = 0, tot_l = 0, tot_i = 0;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) {
            off_l += w < warp ? s_wl[w] : 0;
            off_i += w < warp ? s_wi[w] : 0;
            tot_l += s_wl[w];
            tot_i += s_wi[w];
        }
        if (is_live)
            order_out[base_live + off_l + __popc(bl & below)] = static_cast<int32_t>(r);
        else if (in)
            order_out[base_ign + off_i + __popc(bi & below)] = static_cast<int32_t>(r);
        base_live += tot_l;
        base_ign += tot_i;
        __syncthreads();  // before the next tile overwrites s_wl, s_wi
    }
}

__global__ void __launch_bounds__(kReduceThreads)
    reduce_loss_kernel(const float *loss_rows, const int64_t *labels, int64_t rows,
                       int64_t ignore_index, int reduction, const int64_t *n_in,
                       int64_t *count_into, float *loss_out)
{
    __shared__ int64_t iscratch[kReduceWarps];
    __shared__ double dscratch[kReduceWarps];
    // launched as a dependent of the kernel that wrote the row losses
    grid_dependency_wait();
    // the item count when this call counts (count_into), else a given one
    const bool count = count_into != nullptr;
    int64_t n;
    double total;
    thread_partials(loss_rows, labels, rows, ignore_index, count, n, total);
    block_sum2(n, total, iscratch, dscratch);
    if (threadIdx.x == 0) {
        if (count)
            *count_into = n;
        else
            n = n_in != nullptr ? *n_in : 0;
        double out = total;
        if (reduction == 2)
            out = n > 0 ? total / static_cast<double>(n) : 0.0;
        *loss_out = static_cast<float>(out);
    }
}

cudaError_t launch_count_items(const int64_t *labels, int64_t rows, int64_t ignore_index,
                               int64_t *n_out, int32_t *zero_out, int32_t *order_out,
                               int32_t *order_flag, cudaStream_t stream)
{
    count_items_kernel<<<1, kReduceThreads, 0, stream>>>(labels, rows, ignore_index, n_out,
                                                         zero_out, order_out, order_flag);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_reduce_loss(const float *loss_rows, const int64_t *labels, int64_t rows,
                               int64_t ignore_index, int reduction, const int64_t *n_in,
                               int64_t *count_into, float *loss_out, cudaStream_t stream)
{
    // a programmatic dependent of the row kernel before it: its launch is
    // under way while that kernel finishes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, reduce_loss_kernel, loss_rows, labels, rows,
                                               ignore_index, reduction, n_in, count_into,
                                               loss_out);
    note_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace gbce
