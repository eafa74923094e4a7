// C-ABI entry points of libgbce.so (declared in include/gbce.h): host-side
// argument checks, workspace layout and kernel dispatch.  No entry point
// allocates memory or synchronizes the host.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/gbce.h"
#include "gbce_internal.h"

using gbce::RowParams;

namespace {

std::atomic<uint64_t> g_launches{0};

}  // namespace

void gbce::note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int gbce::device_sm_count()
{
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (dev >= 0 && dev < 64) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0)
            return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

// Few-row problems split the vocabulary so that the row kernel's grid still
// fills the GPU in one wave: rows x splits <= the resident CTAs (3 per SM),
// at most kMaxClusterSplits slices (the portable cluster size, since a split
// row's CTAs form one cluster) of at least kMinSplitElems columns each.
constexpr int kRowCtasPerSm = 3;
constexpr int64_t kMinSplitElems = 8192;
constexpr int64_t kMaxClusterSplits = 8;
constexpr int64_t kMaxVocab = INT32_MAX - 64;  // columns are int32 on the device

int split_count(int64_t rows, int64_t vocab)
{
    if (rows <= 0)
        return 1;
    const int sms = gbce::device_sm_count();
    const int64_t slots = static_cast<int64_t>(kRowCtasPerSm) * (sms > 0 ? sms : 152);
    if (rows * 2 > slots)
        return 1;
    int64_t s = slots / rows;
    if (s > vocab / kMinSplitElems)
        s = vocab / kMinSplitElems;
    if (s > kMaxClusterSplits)
        s = kMaxClusterSplits;
    return s < 1 ? 1 : static_cast<int>(s);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t count = 0;     // int64 n_items scratch
    size_t ticket = 0;    // int32 row ticket of the persistent fused kernel, then the int32
                          // flag of its row order
    size_t loss = 0;      // float [rows] per-row losses
    size_t logp = 0;      // float [rows] per-row log p (two-pass fused calls), or int32
                          // [rows] the persistent kernel's row order
    size_t total = 0;
};

WsLayout ws_layout(int64_t rows, int64_t vocab)
{
    (void)vocab;  // split rows swap their partials on chip, not through the workspace
    WsLayout w;
    if (rows <= 0)
        return w;
    const size_t r = static_cast<size_t>(rows);
    size_t off = 0;
    w.count = off;
    w.ticket = off + 8;
    off += 256;
    w.loss = off;
    off += align_up(r * sizeof(float), 256);
    w.logp = off;
    off += align_up(r * sizeof(float), 256);
    w.total = off;
    return w;
}

size_t elem_size(gbce_dtype dt) { return dt == GBCE_BF16 ? 2 : 4; }

gbce_status check_logits(const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab,
                         int64_t row_stride, float temperature)
{
    if (dtype != GBCE_F32 && dtype != GBCE_BF16)
        return GBCE_EDTYPE;
    if (rows < 0 || vocab < 1 || vocab > kMaxVocab || row_stride < vocab)
        return GBCE_EINVAL;
    if (!(std::isfinite(temperature) && temperature > 0.0f))
        return GBCE_EINVAL;
    if (rows == 0)
        return GBCE_OK;
    if (logits == nullptr)
        return GBCE_EINVAL;
    if (reinterpret_cast<uintptr_t>(logits) % elem_size(dtype) != 0)
        return GBCE_EDTYPE;
    if (row_stride > (INT64_MAX / 8) / rows)
        return GBCE_EINVAL;
    if (rows > INT32_MAX / kMaxClusterSplits)  // grid size: rows x slices CTAs
        return GBCE_EINVAL;
    return GBCE_OK;
}

gbce_status check_workspace(const void *ws, size_t bytes, int64_t rows, int64_t vocab)
{
    const WsLayout w = ws_layout(rows, vocab);
    if (w.total == 0)
        return GBCE_OK;
    if (ws == nullptr || bytes < w.total || reinterpret_cast<uintptr_t>(ws) % 16 != 0)
        return GBCE_EWORKSPACE;
    return GBCE_OK;
}

bool ranges_overlap(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

size_t matrix_bytes(int64_t rows, int64_t vocab, int64_t stride, gbce_dtype dt)
{
    return static_cast<size_t>((rows - 1) * stride + vocab) * elem_size(dt);
}

gbce_status check_dlogits(const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab,
                          int64_t row_stride, const void *dlogits, int64_t d_stride)
{
    if (rows == 0)
        return GBCE_OK;
    if (dlogits == nullptr || d_stride < vocab || d_stride > (INT64_MAX / 8) / rows)
        return GBCE_EINVAL;
    if (reinterpret_cast<uintptr_t>(dlogits) % elem_size(dtype) != 0)
        return GBCE_EDTYPE;
    if (ranges_overlap(logits, matrix_bytes(rows, vocab, row_stride, dtype), dlogits,
                       matrix_bytes(rows, vocab, d_stride, dtype)))
        return GBCE_EINVAL;
    return GBCE_OK;
}

// dlogits row r and logits row r have the same offset modulo 16 bytes for
// every r, so a 16-byte logits vector maps onto a 16-byte dlogits vector.
int same_vector_phase(const void *logits, int64_t row_stride, const void *dlogits,
                      int64_t d_stride, gbce_dtype dt)
{
    const uintptr_t l = reinterpret_cast<uintptr_t>(logits), d = reinterpret_cast<uintptr_t>(dlogits);
    const uint64_t es = elem_size(dt);
    return ((l & 15u) == (d & 15u)) &&
           (((static_cast<uint64_t>(row_stride) * es) & 15u) ==
            ((static_cast<uint64_t>(d_stride) * es) & 15u));
}

// Host check of gbce_ce_options; fills the CE option fields of p.
gbce_status apply_ce_options(const gbce_ce_options *opt, RowParams &p)
{
    p.ls_eps = 0.0f;
    p.dft = 0;
    p.softcap = 0.0f;
    p.inv_cap = 0.0f;
    if (opt == nullptr)
        return GBCE_OK;
    const float eps = opt->label_smoothing;
    if (!(eps >= 0.0f && eps <= 1.0f))  // also rejects NaN
        return GBCE_EINVAL;
    const float cap = opt->softcap;
    if (!(cap >= 0.0f && std::isfinite(cap)))
        return GBCE_EINVAL;
    p.ls_eps = eps;
    p.dft = opt->dft != 0 ? 1 : 0;
    p.softcap = cap;
    p.inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;
    return GBCE_OK;
}

// Statistics and gradient modes of a CE call with these options.
int ce_stats_mode(const RowParams &p)
{
    if (p.softcap > 0.0f)
        return p.ls_eps != 0.0f ? gbce::kModeCeCapSmooth : gbce::kModeCeCap;
    return p.ls_eps != 0.0f ? gbce::kModeCeSmooth : gbce::kModeCe;
}

int ce_grad_mode(const RowParams &p)
{
    return p.softcap > 0.0f ? gbce::kModeGradCap : gbce::kModeGrad;
}

RowParams base_params(const void *logits, gbce_dtype, int64_t rows, int64_t vocab,
                      int64_t row_stride, float temperature, int32_t *dev_status)
{
    RowParams p{};
    p.logits = logits;
    p.rows = rows;
    p.vocab = vocab;
    p.row_stride = row_stride;
    p.T = temperature;
    // log2(e) / T rounded once from the fp64 quotient
    p.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    p.splits = split_count(rows, vocab);
    p.k = 1;
    p.dev_status = dev_status;
    return p;
}

cudaError_t launch_rows(const RowParams &p, gbce_dtype dt, int mode, cudaStream_t s)
{
    return dt == GBCE_BF16 ? gbce::launch_rows<__nv_bfloat16>(p, mode, s)
                           : gbce::launch_rows<float>(p, mode, s);
}

template <typename P>
P *ws_at(void *ws, size_t off)
{
    return reinterpret_cast<P *>(static_cast<char *>(ws) + off);
}

gbce_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GBCE_OK : GBCE_ECUDA; }

}  // namespace

extern "C" {

size_t gbce_workspace_size(int64_t rows, int64_t vocab, int64_t k)
{
    (void)k;  // the workspace holds per-row values only, for any k
    if (rows <= 0 || vocab < 1)
        return 0;
    return ws_layout(rows, vocab).total;
}

uint64_t gbce_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char *gbce_status_string(gbce_status status)
{
    switch (status) {
    case GBCE_OK:
        return "GBCE_OK";
    case GBCE_EINVAL:
        return "GBCE_EINVAL: invalid argument";
    case GBCE_EDTYPE:
        return "GBCE_EDTYPE: unsupported dtype or misaligned element pointer";
    case GBCE_ECUDA:
        return "GBCE_ECUDA: CUDA launch or attribute call failed";
    case GBCE_EWORKSPACE:
        return "GBCE_EWORKSPACE: workspace missing, misaligned or too small";
    }
    return "GBCE: unknown status";
}

gbce_status selective_logsoftmax(const void *logits, gbce_dtype dtype, int64_t rows,
                                 int64_t vocab, int64_t row_stride, const int64_t *index,
                                 int64_t k, float temperature, const uint8_t *row_mask,
                                 float *logp_out, float *entropy_out, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    gbce_status st = check_logits(logits, dtype, rows, vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (k < 1 || k > GBCE_MAX_K)
        return GBCE_EINVAL;
    if (rows == 0)
        return GBCE_OK;
    if (index == nullptr || logp_out == nullptr)
        return GBCE_EINVAL;
    if ((st = check_workspace(workspace, workspace_bytes, rows, vocab)) != GBCE_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    RowParams p = base_params(logits, dtype, rows, vocab, row_stride, temperature, dev_status);
    p.targets = index;
    p.k = k;
    p.row_mask = row_mask;
    p.logp_out = logp_out;
    p.entropy_out = entropy_out;
    const int mode = entropy_out != nullptr ? gbce::kModeLogpEnt : gbce::kModeLogp;
    return cuda_status(launch_rows(p, dtype, mode, s));
}

gbce_status selective_logsoftmax_bwd(const void *logits, gbce_dtype dtype, int64_t rows,
                                     int64_t vocab, int64_t row_stride, const int64_t *index,
                                     int64_t k, float temperature, const uint8_t *row_mask,
                                     const float *grad_logp, const float *saved_logp,
                                     const float *grad_entropy, const float *saved_entropy,
                                     void *dlogits, int64_t dlogits_row_stride,
                                     int32_t *dev_status, void *stream)
{
    gbce_status st = check_logits(logits, dtype, rows, vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (k < 1 || k > GBCE_MAX_K)
        return GBCE_EINVAL;
    if (rows == 0)
        return GBCE_OK;
    if (index == nullptr || grad_logp == nullptr || saved_logp == nullptr)
        return GBCE_EINVAL;
    if ((grad_entropy == nullptr) != (saved_entropy == nullptr))
        return GBCE_EINVAL;
    if ((st = check_dlogits(logits, dtype, rows, vocab, row_stride, dlogits,
                            dlogits_row_stride)) != GBCE_OK)
        return st;

    RowParams p = base_params(logits, dtype, rows, vocab, row_stride, temperature, dev_status);
    p.targets = index;
    p.k = k;
    p.row_mask = row_mask;
    p.dlogits = dlogits;
    p.d_stride = dlogits_row_stride;
    p.vec_store = same_vector_phase(logits, row_stride, dlogits, dlogits_row_stride, dtype);
    p.grad_out = grad_logp;
    p.saved_logp = saved_logp;
    p.grad_entropy = grad_entropy;
    p.saved_entropy = saved_entropy;
    const int mode = grad_entropy != nullptr ? gbce::kModeLogpEntGrad : gbce::kModeLogpGrad;
    return cuda_status(launch_rows(p, dtype, mode, static_cast<cudaStream_t>(stream)));
}

gbce_status ce_fwd(const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab,
                   int64_t row_stride, const int64_t *labels, int64_t ignore_index,
                   float temperature, gbce_reduction reduction,
                   const gbce_ce_options *options, float *loss_out, float *logp_out,
                   float *lse_out, int64_t *n_items_out, void *workspace,
                   size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    RowParams opt_probe{};
    if (apply_ce_options(options, opt_probe) != GBCE_OK)
        return GBCE_EINVAL;
    gbce_status st = check_logits(logits, dtype, rows, vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (reduction != GBCE_NONE && reduction != GBCE_SUM && reduction != GBCE_MEAN)
        return GBCE_EINVAL;
    if ((rows > 0 && (labels == nullptr || loss_out == nullptr)) ||
        (rows == 0 && reduction != GBCE_NONE && loss_out == nullptr))
        return GBCE_EINVAL;
    if ((st = check_workspace(workspace, workspace_bytes, rows, vocab)) != GBCE_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsLayout w = ws_layout(rows, vocab);

    cudaError_t e = cudaSuccess;
    float *loss_rows = loss_out;
    if (rows > 0) {
        if (reduction != GBCE_NONE)
            loss_rows = ws_at<float>(workspace, w.loss);
        RowParams p = base_params(logits, dtype, rows, vocab, row_stride, temperature, dev_status);
        p.targets = labels;
        p.ignore_index = ignore_index;
        p.loss_rows = loss_rows;
        p.logp_out = logp_out;
        p.lse_out = lse_out;
        apply_ce_options(options, p);
        e = launch_rows(p, dtype, ce_stats_mode(p), s);
    }
    int64_t *n_ptr = n_items_out;
    if (n_ptr == nullptr && rows > 0)
        n_ptr = ws_at<int64_t>(workspace, w.count);
    if (e == cudaSuccess && reduction != GBCE_NONE)
        e = gbce::launch_reduce_loss(loss_rows, labels, rows, ignore_index,
                                     static_cast<int>(reduction), nullptr, n_ptr, loss_out, s);
    else if (e == cudaSuccess && n_items_out != nullptr)
        e = gbce::launch_count_items(labels, rows, ignore_index, n_items_out, nullptr, nullptr,
                                     nullptr, s);
    return cuda_status(e);
}

gbce_status ce_bwd(const void *logits, gbce_dtype dtype, int64_t rows, int64_t vocab,
                   int64_t row_stride, const int64_t *labels, int64_t ignore_index,
                   float temperature, gbce_reduction reduction,
                   const gbce_ce_options *options, const float *grad_out,
                   const float *saved_logp, const int64_t *n_items, void *dlogits,
                   int64_t dlogits_row_stride, int32_t *dev_status, void *stream)
{
    RowParams opt_probe{};
    if (apply_ce_options(options, opt_probe) != GBCE_OK)
        return GBCE_EINVAL;
    gbce_status st = check_logits(logits, dtype, rows, vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (reduction != GBCE_NONE && reduction != GBCE_SUM && reduction != GBCE_MEAN)
        return GBCE_EINVAL;
    if (rows == 0)
        return GBCE_OK;
    if (labels == nullptr || grad_out == nullptr || saved_logp == nullptr ||
        (reduction == GBCE_MEAN && n_items == nullptr))
        return GBCE_EINVAL;
    if ((st = check_dlogits(logits, dtype, rows, vocab, row_stride, dlogits,
                            dlogits_row_stride)) != GBCE_OK)
        return st;

    RowParams p = base_params(logits, dtype, rows, vocab, row_stride, temperature, dev_status);
    p.targets = labels;
    p.ignore_index = ignore_index;
    p.dlogits = dlogits;
    p.d_stride = dlogits_row_stride;
    p.vec_store = same_vector_phase(logits, row_stride, dlogits, dlogits_row_stride, dtype);
    p.grad_out = grad_out;
    p.reduction = static_cast<int>(reduction);
    p.n_items = n_items;
    p.saved_logp = saved_logp;
    apply_ce_options(options, p);
    return cuda_status(launch_rows(p, dtype, ce_grad_mode(p), static_cast<cudaStream_t>(stream)));
}

gbce_status ce_fwd_bwd_fused(const void *logits, gbce_dtype dtype, int64_t rows,
                             int64_t vocab, int64_t row_stride, const int64_t *labels,
                             int64_t ignore_index, float temperature,
                             gbce_reduction reduction, const gbce_ce_options *options,
                             const float *grad_out, float *loss_out, float *logp_out,
                             float *lse_out, int64_t *n_items_out, void *dlogits,
                             int64_t dlogits_row_stride, void *workspace,
                             size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    RowParams opt_probe{};
    if (apply_ce_options(options, opt_probe) != GBCE_OK)
        return GBCE_EINVAL;
    gbce_status st = check_logits(logits, dtype, rows, vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (reduction != GBCE_NONE && reduction != GBCE_SUM && reduction != GBCE_MEAN)
        return GBCE_EINVAL;
    if (rows == 0) {
        if (reduction != GBCE_NONE && loss_out == nullptr)
            return GBCE_EINVAL;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaSuccess;
        if (reduction != GBCE_NONE)
            e = gbce::launch_reduce_loss(nullptr, labels, 0, ignore_index,
                                         static_cast<int>(reduction), nullptr, n_items_out,
                                         loss_out, s);
        else if (n_items_out != nullptr)
            e = gbce::launch_count_items(labels, 0, ignore_index, n_items_out, nullptr, nullptr,
                                         nullptr, s);
        return cuda_status(e);
    }
    if (labels == nullptr || loss_out == nullptr || grad_out == nullptr)
        return GBCE_EINVAL;
    if ((st = check_dlogits(logits, dtype, rows, vocab, row_stride, dlogits,
                            dlogits_row_stride)) != GBCE_OK)
        return st;
    if ((st = check_workspace(workspace, workspace_bytes, rows, vocab)) != GBCE_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsLayout w = ws_layout(rows, vocab);
    int64_t *n_ptr = n_items_out != nullptr ? n_items_out : ws_at<int64_t>(workspace, w.count);
    float *loss_rows = reduction == GBCE_NONE ? loss_out : ws_at<float>(workspace, w.loss);

    RowParams p = base_params(logits, dtype, rows, vocab, row_stride, temperature, dev_status);
    // the persistent kernel (all calls but few-row ones) hands out rows from
    // a ticket that the item count zeroes first
    const bool persistent = p.splits == 1;
    p.row_ticket = persistent ? ws_at<int32_t>(workspace, w.ticket) : nullptr;
    // the persistent kernel's row order (live rows first) shares the space
    // of the per-row log p, which only the few-row two-pass path uses
    int32_t *order = persistent ? ws_at<int32_t>(workspace, w.logp) : nullptr;
    int32_t *order_flag = persistent ? ws_at<int32_t>(workspace, w.ticket + 4) : nullptr;
    p.row_order = order;
    p.row_order_flag = order_flag;
    cudaError_t e = cudaSuccess;
    if (reduction == GBCE_MEAN || n_items_out != nullptr || persistent)
        e = gbce::launch_count_items(labels, rows, ignore_index, n_ptr, p.row_ticket, order,
                                     order_flag, s);

    p.targets = labels;
    p.ignore_index = ignore_index;
    p.loss_rows = loss_rows;
    p.logp_out = logp_out;
    p.lse_out = lse_out;
    p.dlogits = dlogits;
    p.d_stride = dlogits_row_stride;
    p.vec_store = same_vector_phase(logits, row_stride, dlogits, dlogits_row_stride, dtype);
    p.grad_out = grad_out;
    p.reduction = static_cast<int>(reduction);
    p.n_items = n_ptr;
    apply_ce_options(options, p);

    if (e == cudaSuccess && (p.softcap == 0.0f || persistent)) {
        // many rows: the persistent kernel (soft-capped or not); few rows:
        // one cluster per row
        e = launch_rows(p, dtype, gbce::kModeFused, s);
    } else if (e == cudaSuccess) {
        // few rows with soft-capped logits: a (split) statistics pass, then
        // a gradient pass
        float *logp_buf = logp_out != nullptr ? logp_out : ws_at<float>(workspace, w.logp);
        p.logp_out = logp_buf;
        e = launch_rows(p, dtype, ce_stats_mode(p), s);
        p.saved_logp = logp_buf;
        if (e == cudaSuccess)
            e = launch_rows(p, dtype, ce_grad_mode(p), s);
    }
    if (e == cudaSuccess && reduction != GBCE_NONE)
        e = gbce::launch_reduce_loss(loss_rows, labels, rows, ignore_index,
                                     static_cast<int>(reduction), n_ptr, nullptr, loss_out, s);
    return cuda_status(e);
}

gbce_status vocab_slice_stats(const void *logits, gbce_dtype dtype, int64_t rows,
                              int64_t slice_vocab, int64_t row_stride, int64_t vocab_offset,
                              int64_t vocab, const int64_t *index, int64_t k,
                              int64_t ignore_index, const uint8_t *row_mask, float temperature,
                              float *partials, int32_t *dev_status, void *stream)
{
    gbce_status st = check_logits(logits, dtype, rows, slice_vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (k < 1 || k > GBCE_MAX_K || vocab_offset < 0 || vocab > kMaxVocab ||
        vocab_offset > vocab - slice_vocab)
        return GBCE_EINVAL;
    if (rows == 0)
        return GBCE_OK;
    if (index == nullptr || partials == nullptr)
        return GBCE_EINVAL;
    RowParams p = base_params(logits, dtype, rows, slice_vocab, row_stride, temperature,
                              dev_status);
    p.targets = index;
    p.k = k;
    p.ignore_index = ignore_index;
    p.row_mask = row_mask;
    p.vocab_offset = vocab_offset;
    p.vocab_total = vocab;
    p.slice_partials = partials;
    return cuda_status(launch_rows(p, dtype, gbce::kModeSliceStats,
                                   static_cast<cudaStream_t>(stream)));
}

gbce_status vocab_slice_combine(const float *partials, int64_t slices,
                                const int64_t *slice_offsets, int64_t rows, const int64_t *index,
                                int64_t k, int64_t ignore_index, const uint8_t *row_mask,
                                float temperature, float *logp_out, float *target_logit_out,
                                float *row_state_out, int32_t *dev_status, void *stream)
{
    if (slices < 1 || slices > GBCE_MAX_SLICES || slice_offsets == nullptr || rows < 0 ||
        k < 1 || k > GBCE_MAX_K || !(std::isfinite(temperature) && temperature > 0.0f))
        return GBCE_EINVAL;
    gbce::SliceOffsets offs{};
    if (slice_offsets[0] != 0 || slice_offsets[slices] > kMaxVocab)
        return GBCE_EINVAL;
    for (int64_t i = 0; i <= slices; ++i) {
        if (i > 0 && slice_offsets[i] <= slice_offsets[i - 1])
            return GBCE_EINVAL;
        offs.off[i] = slice_offsets[i];
    }
    if (rows == 0)
        return GBCE_OK;
    if (partials == nullptr || index == nullptr || logp_out == nullptr)
        return GBCE_EINVAL;
    const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    return cuda_status(gbce::launch_slice_combine(
        partials, static_cast<int>(slices), offs, rows, index, k, ignore_index, row_mask,
        temperature, c, logp_out, target_logit_out, row_state_out, dev_status,
        static_cast<cudaStream_t>(stream)));
}

gbce_status vocab_slice_grad(const void *logits, gbce_dtype dtype, int64_t rows,
                             int64_t slice_vocab, int64_t row_stride, int64_t vocab_offset,
                             int64_t vocab, const int64_t *index, int64_t k, int64_t ignore_index,
                             const uint8_t *row_mask, float temperature, const float *grad_logp,
                             const float *logp, const float *target_logit,
                             const float *row_state, void *dlogits, int64_t dlogits_row_stride,
                             int32_t *dev_status, void *stream)
{
    gbce_status st = check_logits(logits, dtype, rows, slice_vocab, row_stride, temperature);
    if (st != GBCE_OK)
        return st;
    if (k < 1 || k > GBCE_MAX_K || vocab_offset < 0 || vocab > kMaxVocab ||
        vocab_offset > vocab - slice_vocab)
        return GBCE_EINVAL;
    if (rows == 0)
        return GBCE_OK;
    if (index == nullptr || grad_logp == nullptr || logp == nullptr || target_logit == nullptr)
        return GBCE_EINVAL;
    if ((st = check_dlogits(logits, dtype, rows, slice_vocab, row_stride, dlogits,
                            dlogits_row_stride)) != GBCE_OK)
        return st;
    RowParams p = base_params(logits, dtype, rows, slice_vocab, row_stride, temperature,
                              dev_status);
    p.targets = index;
    p.k = k;
    p.ignore_index = ignore_index;
    p.row_mask = row_mask;
    p.vocab_offset = vocab_offset;
    p.vocab_total = vocab;
    p.dlogits = dlogits;
    p.d_stride = dlogits_row_stride;
    p.vec_store = same_vector_phase(logits, row_stride, dlogits, dlogits_row_stride, dtype);
    p.grad_out = grad_logp;
    p.saved_logp = logp;
    p.target_logit = target_logit;
    p.row_state = row_state;
    return cuda_status(launch_rows(p, dtype, gbce::kModeLogpGrad,
                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
