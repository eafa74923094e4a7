// Row kernels for the row-wise log-softmax / cross-entropy path (sm_103a).
//
// One CTA per work unit = (row, vocab slice).  Warp NCW is the producer: its
// lane 0 streams the slice's 16-byte-aligned body through a ring of shared-
// memory stages with 1-D bulk copies (TMA engine, mbarrier completion).  The
// other NCW warps consume each stage: unpack 16-byte vectors, keep an online
// (max, sum) that excludes the target column(s), and -- in the gradient modes
// -- write dlogits with 16-byte streaming stores.  The row's misaligned head
// and tail (when a row does not start on a 16-byte boundary) are read with
// scalar loads.
//
// Sources, by title and section:
//  * the sum that leaves out the target and loss = softplus(log s_others +
//    m - x_y): "Fix softmax collapse in CE, GRPO, KL/JSD and softmax"
//    (Liger-Kernel PR #1555), "Summary";
//  * skipping the target per 16-byte vector instead of per element is the
//    per-block target skip of the unsloth-zoo #2080 commit quoted there
//    ("Fix", forward bullet) at vector granularity: a vector that holds a
//    target takes a masked slow path, every other vector none;
//  * one launch over all rows instead of a chunk loop: "perf(rlhf): chunk
//    selective_log_softmax instead of looping per token", "PR information";
//  * rows with an ignored label are skipped before any read of their
//    logits, and the gradient is g*softmax - g*onehot in a separate buffer:
//    ms-swift PR #10353, "PR information";
//  * a slice split with a later merge of (max, sum) partials: the split
//    partial/combine kernels of the unsloth-zoo #2080 commit ("Fix"), here
//    the CTAs of one thread-block cluster swapping their partials through
//    distributed shared memory instead of a second kernel;
//  * the row entropy taken around the same others' sum, its gradient, label
//    smoothing (the -expm1 label term covers it) and the soft-capped logits
//    of the fused losses' options: the unsloth-zoo #2080 commit ("Fix",
//    "Accuracy"); the DFT row weight: ms-swift PR #10353, "PR information".
#pragma once

#include <atomic>

#include "gbce_device.cuh"
#include "gbce_internal.h"
#include "../../include/gbce.h"

namespace gbce {

constexpr int kConsumerWarps = 8;
constexpr int kChunkBytes = 16384;
constexpr int kStages = 4;
constexpr int kRowThreads = (kConsumerWarps + 1) * 32;
constexpr int kRingBytes = kStages * kChunkBytes;
constexpr int kRingAlign = 128;  // bulk copies need 16-byte aligned shared addresses
constexpr int kDynSmemBytes = kRingBytes + kRingAlign;
constexpr int kMaxClusterCtas = 8;  // portable cluster size limit

struct RowGeom {
    int64_t head;   // scalar elements before the first 16-byte boundary
    int64_t nvec;   // whole 16-byte vectors after them
    int64_t tail0;  // first element after the vectors (scalar tail)
};

template <typename T>
__device__ __forceinline__ RowGeom row_geom(const T *row, int64_t V)
{
    constexpr int VEC = Elem<T>::kVec;
    const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
    int64_t head = static_cast<int64_t>(((16u - mis) & 15u) / sizeof(T));
    if (head > V)
        head = V;
    const int64_t nvec = (V - head) / VEC;
    return {head, nvec, head + nvec * VEC};
}

template <int KMAX>
__device__ __forceinline__ bool is_target(const int32_t (&tg)[KMAX], int32_t col)
{
    bool hit = false;
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
        hit |= (tg[k] == col);
    return hit;
}

// Index of the 16-byte body vector that holds each target column, or -1
// when the column is in the scalar head/tail or the slot is unused.
template <typename T, int KMAX>
__device__ __forceinline__ void target_vectors(const int32_t (&tg)[KMAX], const RowGeom &g,
                                               int32_t (&tv)[KMAX])
{
    constexpr int VEC = Elem<T>::kVec;
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
        tv[k] = (tg[k] >= g.head && tg[k] < g.tail0) ? static_cast<int32_t>((tg[k] - g.head) / VEC)
                                                    : -1;
}

template <int KMAX>
__device__ __forceinline__ bool vector_has_target(const int32_t (&tv)[KMAX], int32_t v)
{
    bool hit = false;
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
        hit |= (tv[k] == v);
    return hit;
}

// The sweep hands body vector vb of a slice [v0, v1) to consumer thread
// (vb - v0) % nc, so each thread knows in advance which of its vectors hold a
// target.  Returns the first such vector of this thread after `after`, or
// INT32_MAX: the sweep then tests one cursor per vector pair instead of K
// indices per vector.
template <int KMAX>
__device__ __forceinline__ int32_t next_target_vector(const int32_t (&tv)[KMAX], int64_t v0,
                                                      int64_t v1, int tid, int nc, int32_t after)
{
    int32_t next = INT32_MAX;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        const int32_t t = tv[k];
        const bool mine = t >= v0 && t < v1 && (t - v0) % nc == tid;
        if (mine && t > after && t < next)
            next = t;
    }
    return next;
}

// Fold one 16-byte vector of logits, masking target columns (slow path).
template <typename T, int KMAX, typename S>
__device__ __forceinline__ void stats_vector(S &st, const uint4 &raw, int32_t col0,
                                             const int32_t (&tg)[KMAX], float c)
{
    constexpr int VEC = Elem<T>::kVec;
    float f[VEC];
    Elem<T>::unpack(raw, f);
    if (S::kSumx)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            st.sumx_add(f[e]);
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        if (is_target<KMAX>(tg, col0 + e))
            f[e] = kNegInf;
    float vmax = f[0];
#pragma unroll
    for (int e = 1; e < VEC; ++e)
        vmax = fmaxf(vmax, f[e]);
    st.add<VEC>(f, vmax, c);
}

// Packed fast paths for vectors that hold no target column.
template <typename T> struct FastVec;

template <> struct FastVec<__nv_bfloat16> {
    __device__ static __forceinline__ uint32_t pmax(const uint4 &a)
    {
        return bf16x2_max(bf16x2_max(a.x, a.y), bf16x2_max(a.z, a.w));
    }
    __device__ static __forceinline__ float unpack_max(uint32_t m)
    {
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    __device__ static __forceinline__ float vmax(const uint4 &a) { return unpack_max(pmax(a)); }
    __device__ static __forceinline__ float vmin(const uint4 &a)
    {
        const uint32_t m = bf16x2_min(bf16x2_min(a.x, a.y), bf16x2_min(a.z, a.w));
        return fminf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    __device__ static __forceinline__ float vmax(const uint4 &a, const uint4 &b)
    {
        return unpack_max(bf16x2_max(pmax(a), pmax(b)));
    }
    template <typename S>
    __device__ static __forceinline__ void add(S &st, const uint4 &a, float c)
    {
        st.add_pairs(bf16x2_to_float2(a.x), bf16x2_to_float2(a.y), c);
        st.add_pairs(bf16x2_to_float2(a.z), bf16x2_to_float2(a.w), c);
    }
};

template <> struct FastVec<float> {
    __device__ static __forceinline__ float vmax(const uint4 &a)
    {
        return fmaxf(fmax3(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z)),
                     __uint_as_float(a.w));
    }
    __device__ static __forceinline__ float vmin(const uint4 &a)
    {
        return fminf(fmin3(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z)),
                     __uint_as_float(a.w));
    }
    __device__ static __forceinline__ float vmax(const uint4 &a, const uint4 &b)
    {
        return fmax3(fmax3(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z)),
                     fmax3(__uint_as_float(a.w), __uint_as_float(b.x), __uint_as_float(b.y)),
                     fmaxf(__uint_as_float(b.z), __uint_as_float(b.w)));
    }
    template <typename S>
    __device__ static __forceinline__ void add(S &st, const uint4 &a, float c)
    {
        st.add_pairs(make_float2(__uint_as_float(a.x), __uint_as_float(a.y)),
                     make_float2(__uint_as_float(a.z), __uint_as_float(a.w)), c);
    }
};

// Soft-capped vectors: z = cap * tanh(x / cap) for a whole 16-byte vector in
// packed pairs.  capped_pairs returns the vector's transformed pairs (4 for
// bf16, 2 for fp32); the caller adds them or writes their gradient.
template <typename T> struct CapVec;

template <> struct CapVec<__nv_bfloat16> {
    static constexpr int kPairs = 4;
    __device__ static __forceinline__ void pairs(const uint4 &a, float2 (&x)[4])
    {
        x[0] = bf16x2_to_float2(a.x);
        x[1] = bf16x2_to_float2(a.y);
        x[2] = bf16x2_to_float2(a.z);
        x[3] = bf16x2_to_float2(a.w);
    }
    __device__ static __forceinline__ uint4 pack(const float2 (&d)[4])
    {
        return make_uint4(float2_to_bf16x2(d[0]), float2_to_bf16x2(d[1]), float2_to_bf16x2(d[2]),
                          float2_to_bf16x2(d[3]));
    }
};

template <> struct CapVec<float> {
    static constexpr int kPairs = 2;
    __device__ static __forceinline__ void pairs(const uint4 &a, float2 (&x)[2])
    {
        x[0] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
        x[1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
    }
    __device__ static __forceinline__ uint4 pack(const float2 (&d)[2])
    {
        return make_uint4(__float_as_uint(d[0].x), __float_as_uint(d[0].y),
                          __float_as_uint(d[1].x), __float_as_uint(d[1].y));
    }
};

// Soft-capping constants of a row pass.  A capped logit is cap * t with
// t = tanh(u), u = x / cap, and in the series range t = u P(u^2) with
// P(s) = 1 + s Q(s) (tanh_poly_pair).  Evaluating P directly in X = x^2
// saves the division by the cap:
//   exponent   capc t = x * A(X),  A = c P(X / cap^2),   coefficients ax
//   value      t      = x * B(X),  B = P(X / cap^2) / cap, coefficients bx
// (capc = cap * c, c = log2(e) / T).  ax[k] and bx[k] scale Q_k by
// cap^-2(k+1), which stays a normal, finite float for caps in
// [2^-13, 2^13]; outside that (no cap in use comes close) every vector takes
// the lane-by-lane path: series_lim = 0.
struct CapConsts {
    float cap, inv_cap, capc, inv_c;
    float series_lim;  // kCapSeriesBound * cap, or 0
    float ax[4], bx[4];
};

__device__ __forceinline__ CapConsts cap_consts(float cap, float inv_cap, float c)
{
    CapConsts k;
    k.cap = cap;
    k.inv_cap = inv_cap;
    k.capc = cap * c;
    k.inv_c = 1.0f / c;
    k.series_lim = (cap >= 0x1p-13f && cap <= 0x1p13f) ? kCapSeriesBound * cap : 0.0f;
    const float i2 = inv_cap * inv_cap;
    const float q[4] = {kTanhQ0, kTanhQ1, kTanhQ2, kTanhQ3};
    float w = i2;
#pragma unroll
    for (int j = 0; j < 4; ++j, w *= i2) {
        k.ax[j] = c * w * q[j];
        k.bx[j] = inv_cap * w * q[j];
    }
    return k;
}

// Whether every logit of a 16-byte vector is inside the series range
// (|x| < series_lim), from its raw max and min.
template <typename T>
__device__ __forceinline__ bool vector_in_series_range(const uint4 &a, float vmax,
                                                       const CapConsts &k)
{
    return fmaxf(vmax, -FastVec<T>::vmin(a)) < k.series_lim;
}

// cap * tanh(x / cap) with CUDA's tanhf, out of line: it is long and the
// sweeps take it only for a running max outside the series range.
static __device__ __noinline__ float capped_tanhf(float x, float cap, float inv_cap)
{
    return cap * tanhf(x * inv_cap);
}

// The capped value of a new running max: the series in its range (the same
// polynomial as the columns it shifts), else tanhf.  Any value close to the
// capped max serves as the shift: the sum is taken relative to it.
__device__ __forceinline__ float capped_max(float x, const CapConsts &k)
{
    const float u = x * k.inv_cap;
    if (fabsf(u) < kCapSeriesBound) {
        const float s = u * u;
        float h = fmaf(kTanhQ3, s, kTanhQ2);
        h = fmaf(h, s, kTanhQ1);
        h = fmaf(h, s, kTanhQ0);
        return k.cap * fmaf(u * s, h, u);
    }
    return capped_tanhf(x, k.cap, k.inv_cap);  // also -inf -> -cap, NaN -> NaN
}

// One vector with a logit outside the series range, lane by lane and out of
// line (so the packed loop stays short): returns the sum of 2^{t capc + nmc}
// and the sum of the capped logits cap * t, t = tanh(x / cap).
template <typename T>
__device__ __noinline__ float2 capped_vector_sums(uint4 a, float inv_cap, float cap, float capc,
                                                  float nmc)
{
    constexpr int VEC = Elem<T>::kVec;
    float f[VEC];
    Elem<T>::unpack(a, f);
    float s = 0.0f, sx = 0.0f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const float t = tanh_lane(f[e] * inv_cap);
        s += ex2(fmaf(t, capc, nmc));
        sx = fmaf(t, cap, sx);
    }
    return make_float2(s, sx);
}

// Raw-max start value of a soft-capped sweep: NaN, so that the first vector
// always raises (a row may open with vectors that are all -inf, whose capped
// value -cap is still a finite max).
__device__ __forceinline__ float capped_sweep_start() { return __uint_as_float(0x7fc00000u); }

// The raw max of one, two or four vectors.
template <typename T, int NV>
__device__ __forceinline__ float raw_vmax(const uint4 (&a)[NV])
{
    static_assert(NV == 1 || NV == 2 || NV == 4, "one, two or four vectors");
    float vmax = NV == 1 ? FastVec<T>::vmax(a[0]) : FastVec<T>::vmax(a[0], a[NV > 1 ? 1 : 0]);
    if (NV == 4)
        vmax = fmaxf(vmax, FastVec<T>::vmax(a[NV - 2], a[NV - 1]));
    return vmax;
}

// Fold NV soft-capped vectors that hold no target (one, or a thread's two
// or four consecutive vectors), whose raw max is vmax.  The running max
// follows the raw max `rise` (vmax, or the max over the warp's lanes: tanh
// is increasing, so the capped max is the cap of the raw max, taken only
// when the raw running max mraw rises).  In the series range each pair's
// exponent is x * A(x^2) - m c (CapConsts), in packed pairs; outside it the
// vectors go lane by lane, and in_range turns false.
template <typename T, int NV, typename S>
__device__ __forceinline__ void stats_capped(S &st, float &mraw, bool &in_range,
                                             const uint4 (&a)[NV], float vmax, float rise,
                                             float c, const CapConsts &k)
{
    constexpr int NP = CapVec<T>::kPairs;
    if (!(rise <= mraw)) {  // a new raw max, the first vector, or NaN (which keeps raising)
        mraw = rise;
        st.raise_to(capped_max(rise, k), c);
    }
    float vmin = FastVec<T>::vmin(a[0]);
#pragma unroll
    for (int v = 1; v < NV; ++v)
        vmin = fminf(vmin, FastVec<T>::vmin(a[v]));
    const bool series = fmaxf(vmax, -vmin) < k.series_lim;
    in_range = in_range && series;
    if (series) {
        const float2 kk = make_float2(st.nmc, st.nmc);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            float2 x[NP];
            CapVec<T>::pairs(a[v], x);
#pragma unroll
            for (int i = 0; i < NP; i += 2) {
                const float2 up = x[i], uq = x[i + 1];
                const float2 ap = tanh_poly_pair(fmul2(up, up), k.ax, c);
                const float2 aq = tanh_poly_pair(fmul2(uq, uq), k.ax, c);
                if (S::kSumx) {
                    const float2 zp = fmul2(up, ap), zq = fmul2(uq, aq);  // capc * t
                    st.add_exponent_pairs(fadd2(zp, kk), fadd2(zq, kk));
                    const float2 ics = make_float2(k.inv_c, k.inv_c);
                    st.sumx_pairs(fmul2(zp, ics), fmul2(zq, ics));
                } else {
                    st.add_exponent_pairs(ffma2(up, ap, kk), ffma2(uq, aq, kk));
                }
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float2 r = capped_vector_sums<T>(a[v], k.inv_cap, k.cap, k.capc, st.nmc);
            st.sa.x += r.x;
            st.sumx_add(r.y);
        }
    }
}

// Fold one soft-capped vector that holds a target column (masked), unpacked.
template <typename T, int KMAX, typename S>
__device__ __forceinline__ void stats_capped_target(S &st, const uint4 &raw, int32_t col0,
                                                    const int32_t (&tg)[KMAX], float c,
                                                    const CapConsts &k)
{
    constexpr int VEC = Elem<T>::kVec;
    float f[VEC];
    Elem<T>::unpack(raw, f);
    float vm = kNegInf;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        f[e] = k.cap * tanhf(f[e] * k.inv_cap);
        st.sumx_add(f[e]);
        if (is_target<KMAX>(tg, col0 + e))
            f[e] = kNegInf;
        vm = fmaxf(vm, f[e]);
    }
    st.template add<VEC>(f, vm, c);
}

// One thread's NPT vectors of a full chunk (thread tid's vectors vb0 + tid +
// u * nc), soft-capped: all four at once when none holds a target (the
// usual case: more independent work between the running-max tests), else
// two at a time, the pair that holds a target (nt) one at a time with the
// target masked.
template <typename T, int KMAX, int NPT, typename S>
__device__ __forceinline__ void stats_capped_chunk(S &st, float &mraw, bool &in_range,
                                                   const uint4 (&raw)[NPT], int32_t vb0,
                                                   int32_t col0, int32_t &nt,
                                                   const int32_t (&tg)[KMAX],
                                                   const int32_t (&tv)[KMAX], int64_t v0,
                                                   int64_t v1, int tid, int nc, bool check,
                                                   float c, const CapConsts &k)
{
    constexpr int VEC = Elem<T>::kVec;
    constexpr int NG = NPT == 4 ? 4 : 2;
    static_assert(NPT % 2 == 0, "vectors go in pairs");
    if (NPT == 4) {
        // the warp's lanes raise the running max together, from a warp-wide
        // max of the lanes whose four vectors hold no target; those lanes
        // fold all four at once
        const bool hit =
            check && static_cast<uint32_t>(nt - (vb0 + tid)) <= static_cast<uint32_t>(3 * nc);
        const uint4(&four)[NG] = reinterpret_cast<const uint4(&)[NG]>(raw);
        const float own = raw_vmax<T, NG>(four);
        const float wmax = warp_max_active(hit ? kNegInf : own);
        if (!hit) {
            stats_capped<T, NG>(st, mraw, in_range, four, own, wmax, c, k);
            return;
        }
    }
#pragma unroll
    for (int u = 0; u < NPT; u += 2) {
        const int32_t va = vb0 + tid + u * nc, vb = va + nc;
        if (check && static_cast<uint32_t>(nt - va) <= static_cast<uint32_t>(vb - va)) {
            stats_capped_target<T, KMAX>(st, raw[u], col0 + va * VEC, tg, c, k);
            stats_capped_target<T, KMAX>(st, raw[u + 1], col0 + vb * VEC, tg, c, k);
            nt = next_target_vector<KMAX>(tv, v0, v1, tid, nc, vb);
            continue;
        }
        const uint4 two[2] = {raw[u], raw[u + 1]};
        const float own = raw_vmax<T, 2>(two);
        stats_capped<T, 2>(st, mraw, in_range, two, own, own, c, k);
    }
}

// Fold body vectors va (and vb, the same thread's next vector) of a row;
// col0 = first column of vector 0; nt = this thread's next target vector
// (next_target_vector), advanced past the vectors a hit folds.
template <typename T, int KMAX, typename S>
__device__ __forceinline__ void stats_one(S &st, const uint4 &a, int32_t va, int32_t col0,
                                          int32_t &nt, const int32_t (&tg)[KMAX], float c,
                                          const int32_t (&tv)[KMAX], int64_t v0, int64_t v1,
                                          int tid, int nc, bool check = true)
{
    constexpr int VEC = Elem<T>::kVec;
    if (check && nt == va) {
        stats_vector<T, KMAX>(st, a, col0 + va * VEC, tg, c);
        nt = next_target_vector<KMAX>(tv, v0, v1, tid, nc, va);
        return;
    }
    if (st.raise_to(FastVec<T>::vmax(a), c))
        FastVec<T>::add(st, a, c);
    else
        st.sumx_add(kNegInf);  // the whole vector is -inf
}

// Two vectors of a full chunk.  With WARP_MAX every lane of the warp folds
// them together: the running max rises for the whole warp at once (one
// warp-wide max, then a uniform raise, where a per-lane max branches apart
// in most groups early in a row -- a gain where many warps share an SM's
// issue slots, a loss of latency where the sweep already runs at the
// bandwidth bound).  A lane whose pair holds a target keeps it out of the
// shared max and folds the pair alone, the target masked.
template <typename T, int KMAX, bool WARP_MAX, typename S>
__device__ __forceinline__ void stats_two(S &st, const uint4 &a, const uint4 &b, int32_t va,
                                          int32_t vb, int32_t col0, int32_t &nt,
                                          const int32_t (&tg)[KMAX], float c,
                                          const int32_t (&tv)[KMAX], int64_t v0, int64_t v1,
                                          int tid, int nc, bool check = true)
{
    constexpr int VEC = Elem<T>::kVec;
    const bool hit = check && static_cast<uint32_t>(nt - va) <= static_cast<uint32_t>(vb - va);
    const float own = hit ? kNegInf : FastVec<T>::vmax(a, b);
    const float wmax = WARP_MAX ? warp_max_active(own) : own;
    if (hit) {
        stats_vector<T, KMAX>(st, a, col0 + va * VEC, tg, c);
        stats_vector<T, KMAX>(st, b, col0 + vb * VEC, tg, c);
        nt = next_target_vector<KMAX>(tv, v0, v1, tid, nc, vb);
        return;
    }
    st.raise_to(wmax, c);
    if (own != kNegInf) {
        FastVec<T>::add(st, a, c);
        FastVec<T>::add(st, b, c);
    } else {
        st.sumx_add(kNegInf);  // both vectors are -inf
    }
}

// h = sum 2^z z (z = x c - m c, target columns left out) over the columns
// one consumer thread swept -- its share of the head and tail, and the body
// vectors vb with (vb - v0) % nc == tid -- re-read from global memory with
// -inf logits adding 0.  Taken only by a thread whose packed h went NaN on a
// -inf logit while its sum stayed finite.
template <typename T, int KMAX>
__device__ __forceinline__ float rescan_entropy_moment(const T *row, const RowGeom &g, int64_t V,
                                                   int64_t v0, int64_t v1, bool first, bool last,
                                                   const int32_t (&tg)[KMAX], float c, float nmc,
                                                   int tid, int nc)
{
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    using S = OnlineStats<true>;
    float h = 0.0f;
    const auto term = [&](float x, int64_t col) {
        if (!is_target<KMAX>(tg, static_cast<int32_t>(col))) {
            const float z = fmaf(x, c, nmc);
            h = fmaf(ex2(z), S::zfin(z), h);
        }
    };
    if (first)
        for (int64_t e = tid; e < g.head; e += nc)
            term(E::load(row + e), e);
    if (last)
        for (int64_t e = g.tail0 + tid; e < V; e += nc)
            term(E::load(row + e), e);
    const uint4 *body = reinterpret_cast<const uint4 *>(row + g.head);
    for (int64_t vb = v0 + tid; vb < v1; vb += nc) {
        float f[VEC];
        E::unpack(body[vb], f);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            term(f[e], g.head + vb * VEC + e);
    }
    return h;
}

// ------------------------------------------- whole-row passes (off the hot path)
//
// A few rows need a second look at all of their columns after (or before)
// the pipelined sweep: the entropy of a confident row whose dominant column
// is not the reference column.  These passes read the row from global
// memory (16-byte vectors for the aligned body) with every consumer thread
// of the CTA and synchronize on named barrier 1; they never run for the
// other rows.

// Calls f(x, col) for every column that consumer thread `tid` of `nc` owns
// in a whole-row pass: its share of the scalar head and tail, and the body
// vectors tid, tid + nc, ...
template <typename T, typename F>
__device__ __forceinline__ void for_each_own_column(const T *row, const RowGeom &g, int64_t V,
                                                    int tid, int nc, F &&f)
{
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    for (int64_t e = tid; e < g.head; e += nc)
        f(E::load(row + e), e);
    for (int64_t e = g.tail0 + tid; e < V; e += nc)
        f(E::load(row + e), e);
    const uint4 *body = reinterpret_cast<const uint4 *>(row + g.head);
    for (int64_t vb = tid; vb < g.nvec; vb += nc) {
        float v[VEC];
        E::unpack(ld_nc_v4(body + vb), v);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            f(v[e], g.head + vb * VEC + e);
    }
}

// The largest logit M of a row and the first column d holding it, found by
// NCW consumer warps together (NCW == 1: one warp, no shared memory or
// barrier); every participating thread gets both.
template <typename T, int NCW>
__device__ void row_argmax(const T *row, const RowGeom &g, int64_t V, int tid, float *red_m,
                           int32_t *red_i, float &M, int32_t &d)
{
    constexpr int NC = NCW * 32;
    const int warp = tid >> 5, lane = tid & 31;
    const auto better = [](float xa, int32_t ia, float xb, int32_t ib) {
        return xb > xa || (xb == xa && ib < ia);
    };
    float bm = kNegInf;
    int32_t bi = INT32_MAX;
    for_each_own_column<T>(row, g, V, tid, NC, [&](float x, int64_t col) {
        if (better(bm, bi, x, static_cast<int32_t>(col))) {
            bm = x;
            bi = static_cast<int32_t>(col);
        }
    });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, bm, off);
        const int32_t i2 = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(bm, bi, m2, i2)) {
            bm = m2;
            bi = i2;
        }
    }
    if (NCW == 1) {
        M = bm;
        d = bi;
        return;
    }
    if (lane == 0) {
        red_m[warp] = bm;
        red_i[warp] = bi;
    }
    named_sync(1, NC);
    bm = kNegInf;
    bi = INT32_MAX;
    for (int w = 0; w < NCW; ++w)
        if (better(bm, bi, red_m[w], red_i[w])) {
            bm = red_m[w];
            bi = red_i[w];
        }
    named_sync(1, NC);  // the scratch arrays are free again
    M = bm;
    d = bi;
}

// Entropy of a row with column d (logit xd) as the reference column of
// finalize_entropy: the state (m, s, h) of every other column from a
// whole-row pass by NCW warps (NCW == 1: one warp, no shared memory or
// barrier).  For a confident row whose dominant column d is not the column
// the sweep left out, this is what keeps 1 - p_d (and so the entropy) from
// rounding: the sweep's s = 1 + (everything else) cannot hold the rest when
// it is below fp32's resolution at 1.  Valid in thread 0 of the group.
template <typename T, int NCW>
__device__ float entropy_around(const T *row, const RowGeom &g, int64_t V, int32_t d, float xd,
                                float c, float temperature, int tid, float *red_m, float *red_s,
                                float *red_h)
{
    constexpr int NC = NCW * 32;
    const int warp = tid >> 5, lane = tid & 31;
    OnlineStats<true> st;
    for_each_own_column<T>(row, g, V, tid, NC,
                           [&](float x, int64_t col) { st.add1(col == d ? kNegInf : x, c); });
    float m = st.m, s = st.sum(), h = st.hsum();
    warp_merge_state<kHMoment>(m, s, h, c, st.residual(c));
    if (NCW == 1)
        return finalize_entropy(m, s, h, xd, temperature);
    if (lane == 0) {
        red_m[warp] = m;
        red_s[warp] = s;
        red_h[warp] = h;
    }
    named_sync(1, NC);
    float H = 0.0f;
    if (warp == 0) {
        m = lane < NCW ? red_m[lane] : kNegInf;
        s = lane < NCW ? red_s[lane] : 0.0f;
        h = lane < NCW ? red_h[lane] : 0.0f;
        warp_merge_state<kHMoment>(m, s, h, c);
        H = finalize_entropy(m, s, h, xd, temperature);
    }
    named_sync(1, NC);
    return H;
}

// The whole row's max M and its sum S = sum_j 2^{(x_j - M) c} (x_j capped
// under CAP), from NCW consumer warps reading the row from global memory
// (all of them take part; every one gets both).  For a backward whose
// gathered column lies far below the row's max (rebase_grad_consts): a
// second read of that rare row.
template <typename T, int NCW, bool CAP>
__device__ void row_max_sum(const T *row, const RowGeom &g, int64_t V, int tid, float c,
                            float cap, float inv_cap, float *red_m, float *red_s, float &M,
                            float &S)
{
    constexpr int NC = NCW * 32;
    const int warp = tid >> 5, lane = tid & 31;
    OnlineStats<false> st;
    for_each_own_column<T>(row, g, V, tid, NC, [&](float x, int64_t) {
        st.add1(CAP ? cap * tanhf(x * inv_cap) : x, c);
    });
    float m = st.m, s = st.sum(), h = 0.0f;
    warp_merge_state<kHNone>(m, s, h, c, st.residual(c));
    if (lane == 0) {
        red_m[warp] = m;
        red_s[warp] = s;
    }
    named_sync(1, NC);
    m = lane < NCW ? red_m[lane] : kNegInf;
    s = lane < NCW ? red_s[lane] : 0.0f;
    warp_merge_state<kHNone>(m, s, h, c);
    named_sync(1, NC);  // the scratch arrays are free again
    M = m;
    S = s;
}

// Q = sum_{j != d} p_j (x_d - x_j) / T over a row, with p_j = exp((x_j - x_t)/T
// + log p_t) taken from a column t whose log p is known accurately.  For the
// dominant column d, Q equals H + log p_d (H the row entropy), but as a sum
// of non-negative terms: the gradient of the entropy at d needs that value,
// and H + log p_d cancels when p_d is near 1.  Every consumer thread gets Q.
template <typename T, int NCW>
__device__ float entropy_gap(const T *row, const RowGeom &g, int64_t V, int32_t d, float xd,
                             float xref, float lref2, float c, float inv_t, int tid, float *red)
{
    constexpr int NC = NCW * 32;
    const int warp = tid >> 5, lane = tid & 31;
    // 2^(z + 32), z = log2 p_j from a reference column (x_ref, log2 p_ref):
    // p_j down to 2^-158 although ex2 flushes below 2^-126
    const float kb = lref2 + 32.0f;
    float acc = 0.0f;
    for_each_own_column<T>(row, g, V, tid, NC, [&](float x, int64_t col) {
        if (col != d) {
            const float pj = ex2(fmaf(x - xref, c, kb));
            if (pj > 0.0f || pj != pj)  // a -inf logit adds 0 (not 0 * inf); NaN stays
                acc = fmaf(pj, (xd - x) * inv_t, acc);
        }
    });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    if (lane == 0)
        red[warp] = acc;
    named_sync(1, NC);
    float q = 0.0f;
    for (int w = 0; w < NCW; ++w)
        q += red[w];
    named_sync(1, NC);
    return q * 0x1p-32f;
}

// Per-row constants of the gradient pass.  The exponent carries an offset
// of +32 that g/T takes back as 2^-32, so that entries far below 2^-126
// (confident rows) come out as exact fp32 subnormals although ex2 itself
// flushes subnormal results; |g/T| < 2^-90 skips the offset.
struct GradConsts {
    float nxy;  // -x_ref (x_y, or the row max after rebase_grad_consts)
    float c;    // log2(e) / T
    float kb;   // log2 p_ref + offset
    float kbx;  // kb - x_ref * c: the bf16 path's exponent is x * c + kbx
    float off;  // the offset: 32 or 0
    float gs;   // g / T * 2^-offset
    float dy;   // g / T * expm1(log p), the label column
    float c0;   // constant added to every non-label element (label smoothing)
    // entropy gradient: an element is 2^z (ea + eb z) instead of gs 2^z
    float ea, eb;
};

__device__ __forceinline__ GradConsts grad_consts(float xy, float c, float logp, float gscale)
{
    const bool offset = fabsf(gscale) >= 0x1p-90f;
    GradConsts k;
    k.nxy = -xy;
    k.c = c;
    k.off = offset ? 32.0f : 0.0f;
    k.kb = fmaf(logp, kLog2e, k.off);
    k.kbx = fmaf(-xy, c, k.kb);
    k.gs = offset ? gscale * 0x1p-32f : gscale;
    k.dy = gscale * expm1f(logp);
    k.c0 = 0.0f;
    k.ea = k.eb = 0.0f;
    return k;
}

// Every gradient element evaluates z_j = log2 p_j + off as (x_j - x_ref) c +
// log2 p_ref + off.  With the gathered column as the reference (x_y and the
// forward's log p_y), a column far above it gets z_j as the sum of two large
// numbers of opposite sign, which leaves it an error of about 2^-24 times
// their size: past ~40 nats, more than the gradient's fp32 bound.  Moved to
// the row's max M with log2 p_M = -log2 S (S, the row's sum relative to M,
// lies in [1, V]), the dominant column's z is exact to rounding and every
// other column's error is that of its own distance below M.
__device__ __forceinline__ void rebase_grad_consts(GradConsts &k, float M, float S)
{
    if (!(S > 0.0f) || !isfinite(M))  // (an empty or NaN row: nothing to gain)
        return;
    k.nxy = -M;
    k.kb = k.off - log2f(S);
    k.kbx = fmaf(-M, k.c, k.kb);
}

// A vocabulary slice's gradient: the row is not all here, so its whole
// state comes from the combine (RowParams::row_state) instead of a re-read.
__device__ __forceinline__ bool slice_row(const RowParams &p) { return p.vocab_total > 0; }

// Gathered log p below which the standalone backwards first read the row's
// max and sum (row_max_sum) to rebase their constants: with the gathered
// reference, the error of a dominant column's gradient grows as 2^-24 times
// (|log p| + its margin); below this it could pass the fp32 bound.
constexpr float kRebaseLogp = -40.0f;

// The (max, sum) state of a row that a fused call's statistics left over
// its non-target columns (m, s), with the target logit xt folded in: the
// row's max M and S = sum_j 2^{(x_j - M) c}.
__device__ __forceinline__ void row_state_with_target(float m, float s, float xt, float c,
                                                      float &M, float &S)
{
    M = fmaxf(m, xt);
    S = (m == kNegInf ? 0.0f : s * ex2((m - M) * c)) + (xt == kNegInf ? 0.0f : ex2((xt - M) * c));
}

// Loss of one kept row of the token CE from log p_y, x_y and (label
// smoothing) the row's sum of logits: w ((1 - eps)(-log p_y) + eps (lse -
// mean_j z_j)), lse = x_y / T - log p_y, w = p_y under DFT, else 1.
__device__ __forceinline__ float ce_row_loss(float lp, float xy, float sumx, float T, float eps,
                                             int dft, int64_t V)
{
    float loss = -lp;
    if (eps != 0.0f) {
        const float lse = xy / T - lp;
        const float mean_z = sumx / (T * static_cast<float>(V));
        loss = fmaf(1.0f - eps, -lp, eps * (lse - mean_z));
    }
    return dft ? expf(lp) * loss : loss;
}

// Gradient constants of a kept CE row with upstream g: every element is
// (g w / T)(p_j - eps / V), the label's (g w / T)(expm1(log p_y) + eps - eps / V),
// w = p_y under DFT (held constant), else 1.
__device__ __forceinline__ GradConsts grad_consts_ce(float xy, float c, float logp, float g,
                                                     float T, float eps, int dft, int64_t V)
{
    // (g / T) first: with a DFT weight below fp32's normal range, g p_y
    // could round to 0 where (g / T) p_y is still a subnormal
    const float gscale = dft ? (g / T) * expf(logp) : g / T;
    GradConsts k = grad_consts(xy, c, logp, gscale);
    if (eps != 0.0f) {
        const float u = eps / static_cast<float>(V);
        k.c0 = -gscale * u;
        k.dy = gscale * (expm1f(logp) + (eps - u));
    }
    return k;
}

// Constants for a gradient whose element j != gathered columns is
// p_j (A + B log p_j) -- the selective log-softmax gradient (A = -G/T, B = 0)
// plus the entropy's (A -= gH H / T, B = -gH / T).  With z = log2 p_j + off
// (the exponent the element evaluates), log p_j = (z - off) ln 2, so the
// element is 2^z * 2^-off (A - B off ln2 + B ln2 z) = 2^z (ea + eb z).
__device__ __forceinline__ GradConsts grad_consts_ent(float xy, float c, float logp, float A,
                                                      float B)
{
    // same offset rule as grad_consts, on the larger coefficient
    const float big = fmaxf(fabsf(A), fabsf(B));
    GradConsts k = grad_consts(xy, c, logp, big);
    const bool offset = big >= 0x1p-90f;
    const float off = offset ? 32.0f : 0.0f, scale = offset ? 0x1p-32f : 1.0f;
    constexpr float kLn2 = 0.69314718055994531f;
    k.ea = scale * fmaf(-B * kLn2, off, A);
    k.eb = scale * (B * kLn2);
    return k;
}

// dlogits of one element j != y: g/T * exp((x_j - x_y)/T + log p).
__device__ __forceinline__ float grad_scalar(float x, const GradConsts &k)
{
    return fmaf(k.gs, ex2(fmaf(x + k.nxy, k.c, k.kb)), k.c0);
}

// The same element with the entropy term: 2^z (ea + eb z); a -inf logit
// (2^z = 0) gives 0, not 0 * inf.
__device__ __forceinline__ float grad_scalar_ent(float x, const GradConsts &k)
{
    const float z = fmaf(x + k.nxy, k.c, k.kb);
    return ex2(z) * fmaf(k.eb, OnlineStats<true>::zfin(z), k.ea);
}

// dlogits of one 16-byte vector.  yoff = label column - first column of
// the vector; only the one vector of a row that holds the label (unsigned
// yoff < VEC) takes the patch branch.  run() returns the packed vector;
// run_unpacked() the fp32 values, for stores that cannot be 16-byte.
template <typename T> struct GradVec;

template <> struct GradVec<__nv_bfloat16> {
    // bf16 logits are exact in fp32 and |x c| is small, so x c + (kb - x_y c)
    // in one fused multiply-add stays within a few fp32 ulps of the exponent.
    template <bool ENT = false>
    __device__ static __forceinline__ uint4 run(const uint4 &raw, int32_t yoff, const GradConsts &k)
    {
        const float2 cc = make_float2(k.c, k.c), kk = make_float2(k.kbx, k.kbx);
        const float2 gg = make_float2(k.gs, k.gs), c0 = make_float2(k.c0, k.c0);
        const float2 ea = make_float2(k.ea, k.ea), eb = make_float2(k.eb, k.eb);
        const auto one = [&](uint32_t w) {
            const float2 z = ffma2(bf16x2_to_float2(w), cc, kk);
            const float2 e = make_float2(ex2(z.x), ex2(z.y));
            if (ENT) {
                using S = OnlineStats<true>;
                const float2 wv = ffma2(make_float2(S::zfin(z.x), S::zfin(z.y)), eb, ea);
                return float2_to_bf16x2(fmul2(e, wv));
            }
            return float2_to_bf16x2(ffma2(e, gg, c0));
        };
        uint4 o = make_uint4(one(raw.x), one(raw.y), one(raw.z), one(raw.w));
        if (static_cast<uint32_t>(yoff) < 8u) {
            const uint32_t dyb = __bfloat16_as_ushort(__float2bfloat16_rn(k.dy));
            const bool hi = (yoff & 1) != 0;
            const auto patch = [&](uint32_t v) {
                return hi ? ((v & 0x0000ffffu) | (dyb << 16)) : ((v & 0xffff0000u) | dyb);
            };
            const int pair = yoff >> 1;
            o.x = pair == 0 ? patch(o.x) : o.x;
            o.y = pair == 1 ? patch(o.y) : o.y;
            o.z = pair == 2 ? patch(o.z) : o.z;
            o.w = pair == 3 ? patch(o.w) : o.w;
        }
        return o;
    }
    template <bool ENT = false>
    __device__ static __forceinline__ void run_unpacked(const uint4 &raw, int32_t yoff,
                                                        const GradConsts &k, float (&d)[8])
    {
        float f[8];
        Elem<__nv_bfloat16>::unpack(raw, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float z = fmaf(f[e], k.c, k.kbx);
            const float v = ENT ? ex2(z) * fmaf(k.eb, OnlineStats<true>::zfin(z), k.ea)
                                : fmaf(k.gs, ex2(z), k.c0);
            d[e] = (e == yoff) ? k.dy : v;
        }
    }
};

template <> struct GradVec<float> {
    template <bool ENT = false>
    __device__ static __forceinline__ uint4 run(const uint4 &raw, int32_t yoff, const GradConsts &k)
    {
        const float2 nn = make_float2(k.nxy, k.nxy), cc = make_float2(k.c, k.c);
        const float2 kk = make_float2(k.kb, k.kb), gg = make_float2(k.gs, k.gs);
        const float2 p0 = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
        const float2 p1 = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
        const float2 z0 = ffma2(fadd2(p0, nn), cc, kk), z1 = ffma2(fadd2(p1, nn), cc, kk);
        float2 g0 = gg, g1 = gg;
        const float2 c0 = make_float2(k.c0, k.c0);
        if (ENT) {
            using S = OnlineStats<true>;
            const float2 ea = make_float2(k.ea, k.ea), eb = make_float2(k.eb, k.eb);
            g0 = ffma2(make_float2(S::zfin(z0.x), S::zfin(z0.y)), eb, ea);
            g1 = ffma2(make_float2(S::zfin(z1.x), S::zfin(z1.y)), eb, ea);
        }
        const float2 d0 = ffma2(make_float2(ex2(z0.x), ex2(z0.y)), g0, c0);
        const float2 d1 = ffma2(make_float2(ex2(z1.x), ex2(z1.y)), g1, c0);
        uint4 o = make_uint4(__float_as_uint(d0.x), __float_as_uint(d0.y), __float_as_uint(d1.x),
                             __float_as_uint(d1.y));
        if (static_cast<uint32_t>(yoff) < 4u) {
            const uint32_t dyb = __float_as_uint(k.dy);
            o.x = yoff == 0 ? dyb : o.x;
            o.y = yoff == 1 ? dyb : o.y;
            o.z = yoff == 2 ? dyb : o.z;
            o.w = yoff == 3 ? dyb : o.w;
        }
        return o;
    }
    template <bool ENT = false>
    __device__ static __forceinline__ void run_unpacked(const uint4 &raw, int32_t yoff,
                                                        const GradConsts &k, float (&d)[4])
    {
        float f[4];
        Elem<float>::unpack(raw, f);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            d[e] = (e == yoff) ? k.dy : (ENT ? grad_scalar_ent(f[e], k) : grad_scalar(f[e], k));
    }
};

// grad_capped for a vector with a logit outside the series range, lane by
// lane and out of line: fma(gs, 2^z, c0) * (1 - t^2), z = t * capc + kbx,
// the chain factor from tanh_chain.
template <typename T>
__device__ __noinline__ uint4 grad_capped_lanes(uint4 a, float inv_cap, float capc, float kbx,
                                                float gs, float c0)
{
    constexpr int VEC = Elem<T>::kVec;
    float f[VEC];
    Elem<T>::unpack(a, f);
    float d[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const float u = f[e] * inv_cap;
        float unscale;
        const float chain = tanh_chain(u, unscale);
        d[e] = (fmaf(gs, ex2(fmaf(tanh_lane(u), capc, kbx)), c0) * chain) * unscale;
    }
    return Elem<T>::pack(d);
}

// The soft-capped gradient of the vector that holds the label (element
// yoff), lane by lane with tanhf and out of line (once per row): the label
// element is dy * (1 - t^2), the others as in grad_capped_lanes, the chain
// factor from tanh_chain.
template <typename T>
__device__ __noinline__ uint4 grad_capped_label_vector(uint4 a, int32_t yoff, float dy,
                                                       float inv_cap, float capc, float kbx,
                                                       float gs, float c0)
{
    constexpr int VEC = Elem<T>::kVec;
    float f[VEC];
    Elem<T>::unpack(a, f);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const float u = f[e] * inv_cap;
        float unscale;
        const float chain = tanh_chain(u, unscale);
        const float d = e == yoff ? dy : fmaf(gs, ex2(fmaf(tanhf(u), capc, kbx)), c0);
        f[e] = (d * chain) * unscale;
    }
    return Elem<T>::pack(f);
}

// Gradient of one soft-capped vector without the label whose logits are
// all inside the series range, packed: element j is fma(gs, 2^z, c0) *
// (1 - t^2), t = tanh(x_j / cap) = x_j B(x_j^2) (CapConsts), with the
// exponent z = t * capc + kbx of the uncapped formula on the capped logit
// (kbx from the capped label logit), evaluated as (-gs 2^z - c0)(t^2 - 1):
// the sign goes into the constants, so the chain factor is one fused
// multiply-add (|t| < 0.5 in this range: t^2 - 1 cancels nothing).
template <typename T>
__device__ __forceinline__ uint4 grad_capped_series(const uint4 &a, const GradConsts &k,
                                                    const CapConsts &cp)
{
    constexpr int NP = CapVec<T>::kPairs;
    float2 x[NP];
    CapVec<T>::pairs(a, x);
    const float2 cc = make_float2(cp.capc, cp.capc), kk = make_float2(k.kbx, k.kbx);
    const float2 ngs = make_float2(-k.gs, -k.gs), nc0 = make_float2(-k.c0, -k.c0);
    const float2 m1 = make_float2(-1.0f, -1.0f);
    float2 d[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const float2 t = fmul2(x[i], tanh_poly_pair(fmul2(x[i], x[i]), cp.bx, cp.inv_cap));
        const float2 z = ffma2(t, cc, kk);
        const float2 e = make_float2(ex2(z.x), ex2(z.y));
        d[i] = fmul2(ffma2(e, ngs, nc0), ffma2(t, t, m1));
    }
    return CapVec<T>::pack(d);
}

// Gradient of one soft-capped vector without the label: packed in the
// series range, else lane by lane.
template <typename T>
__device__ __forceinline__ uint4 grad_capped(const uint4 &a, const GradConsts &k,
                                             const CapConsts &cp)
{
    if (vector_in_series_range<T>(a, FastVec<T>::vmax(a), cp))
        return grad_capped_series<T>(a, k, cp);
    return grad_capped_lanes<T>(a, cp.inv_cap, cp.capc, k.kbx, k.gs, k.c0);
}

// The soft-capped gradient of one thread's NPT vectors of a full chunk
// (vectors tid + u * nc, the label at column offset ybase of the chunk),
// stored with 16-byte streaming stores.  One range test covers all NPT
// vectors, and none is needed when the statistics pass already found every
// logit of the row inside the series range (row_in_range).
template <typename T, int NPT>
__device__ __forceinline__ void grad_capped_chunk(const uint4 *chunk, T *dbase, int32_t ybase,
                                                  int tid, int nc, bool row_in_range,
                                                  const GradConsts &k, const CapConsts &cp)
{
    constexpr int VEC = Elem<T>::kVec;
    uint4 raw[NPT];
#pragma unroll
    for (int u = 0; u < NPT; ++u)
        raw[u] = chunk[tid + u * nc];
    bool series = row_in_range;
    if (!series) {
        float vmax = FastVec<T>::vmax(raw[0]), vmin = FastVec<T>::vmin(raw[0]);
#pragma unroll
        for (int u = 1; u < NPT; ++u) {
            vmax = fmaxf(vmax, FastVec<T>::vmax(raw[u]));
            vmin = fminf(vmin, FastVec<T>::vmin(raw[u]));
        }
        series = fmaxf(vmax, -vmin) < cp.series_lim;
    }
#pragma unroll
    for (int u = 0; u < NPT; ++u) {
        const int v = tid + u * nc;
        const int32_t yoff = ybase - v * VEC;
        uint4 d;
        if (static_cast<uint32_t>(yoff) < static_cast<uint32_t>(VEC))
            d = grad_capped_label_vector<T>(raw[u], yoff, k.dy, cp.inv_cap, cp.capc, k.kbx,
                                            k.gs, k.c0);
        else if (series)
            d = grad_capped_series<T>(raw[u], k, cp);
        else
            d = grad_capped_lanes<T>(raw[u], cp.inv_cap, cp.capc, k.kbx, k.gs, k.c0);
        st_cs_v4(dbase + v * VEC, d);
    }
}

// log p of target k, whose "others" are every column outside the target set
// S (already folded into (mS, sS)) plus the distinct members of S other
// than target k itself.
template <int KMAX>
__device__ __forceinline__ float logp_with_targets(float mS, float sS, const int32_t *tg,
                                                   const float *xt, int K, int k, float c,
                                                   float T)
{
    float m = mS, s = sS;
    const int32_t tk = tg[k];
    for (int j = 0; j < K; ++j) {
        const int32_t tj = tg[j];
        if (tj < 0 || tj == tk)
            continue;
        bool dup = false;
        for (int i = 0; i < j; ++i)
            dup |= (tg[i] == tj);
        if (!dup)
            merge_max_sum(m, s, xt[j], 1.0f, c);
    }
    return finalize_logp(m, s, xt[k], T);
}

// Entropy of a row from the state (mS, sS, hS) of every column outside the
// target set S: the distinct members of S other than the first index are
// folded in, and the first index is the reference column of
// finalize_entropy.  That is accurate to fp32 rounding unless the row is
// confident in another column d: the others' max m lies above x_t0 and the
// others' sum s = 1 + rest (d's own term is the 1) has rest < 2^-5.  Then
// 1 + rest keeps only the rest's leading digits, the entropy (about rest *
// log(1/rest)) inherits their loss, and the caller recomputes it around d
// (entropy_around).  With rest >= 2^-5 the absolute error of log s, about
// 1e-7, stays below 1e-5 of the entropy.  NaN when the first index is out
// of range.
template <int KMAX>
__device__ __forceinline__ float entropy_with_targets(float mS, float sS, float hS,
                                                      const int32_t *tg, const float *xt, int K,
                                                      float c, float T, bool &rescan)
{
    const int32_t t0 = tg[0];
    rescan = false;
    if (t0 < 0)
        return __int_as_float(0x7fc00000);
    float m = mS, s = sS, h = hS;
    for (int j = 1; j < K; ++j) {
        const int32_t tj = tg[j];
        if (tj < 0 || tj == t0)
            continue;
        bool dup = false;
        for (int i = 1; i < j; ++i)
            dup |= (tg[i] == tj);
        if (!dup)
            merge_max_sum_h(m, s, h, xt[j], 1.0f, 0.0f, c);
    }
    rescan = m > xt[0] && s < 1.03125f && isfinite(m);
    return finalize_entropy(m, s, h, xt[0], T);
}

__device__ __forceinline__ float upstream_grad(const RowParams &p, int64_t r)
{
    if (p.reduction == 0)
        return p.grad_out[r];
    if (p.reduction == 1)
        return p.grad_out[0];
    const int64_t n = *p.n_items;
    return n > 0 ? p.grad_out[0] / static_cast<float>(n) : 0.0f;
}

__device__ __forceinline__ void report(int32_t *dev_status, int bits)
{
    if (dev_status != nullptr)
        atomicOr(dev_status, bits);
}

// Fill this unit's slice of a dlogits row with `value` (0 for an ignored
// row, NaN for a bad label), using every thread of the CTA.
template <typename T>
__device__ void fill_row_slice(T *drow, int64_t V, int split, int splits, float value)
{
    constexpr int VEC = Elem<T>::kVec;
    const RowGeom g = row_geom<T>(drow, V);
    const int64_t v0 = g.nvec * split / splits, v1 = g.nvec * (split + 1) / splits;
    float f[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        f[e] = value;
    const uint4 pat = Elem<T>::pack(f);
    uint4 *body = reinterpret_cast<uint4 *>(drow + g.head);
    for (int64_t v = v0 + threadIdx.x; v < v1; v += blockDim.x)
        st_cs_v4(body + v, pat);
    if (split == 0)
        for (int64_t e = threadIdx.x; e < g.head; e += blockDim.x)
            Elem<T>::store(drow + e, value);
    if (split == splits - 1)
        for (int64_t e = g.tail0 + threadIdx.x; e < V; e += blockDim.x)
            Elem<T>::store(drow + e, value);
}

template <typename T, int MODE, int KMAX>
__global__ void __launch_bounds__(kRowThreads, (MODE != kModeFused && KMAX <= 4) ? 3 : 2)
    row_kernel(const RowParams p)
{
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    constexpr int NCW = kConsumerWarps;
    constexpr int NC = NCW * 32;
    constexpr int CV = kChunkBytes / 16;  // vectors per full chunk
    constexpr int PER_THREAD = CV / NC;
    static_assert(CV % NC == 0, "chunk must split evenly over consumer threads");
    constexpr bool kSelGrad = (MODE == kModeLogpGrad || MODE == kModeLogpEntGrad);
    constexpr bool kEntGrad = (MODE == kModeLogpEntGrad);
    constexpr bool kCeGrad = (MODE == kModeGrad || MODE == kModeGradCap);  // ce_bwd
    constexpr bool kCap = (MODE == kModeCeCap || MODE == kModeCeCapSmooth ||
                           MODE == kModeGradCap);  // soft-capped logits
    constexpr bool kStats = (!kCeGrad && !kSelGrad);
    constexpr bool kGrad = (kCeGrad || MODE == kModeFused || kSelGrad);
    constexpr bool kEnt = (MODE == kModeLogpEnt);                  // + row entropy
    constexpr bool kLogpFwd = (MODE == kModeLogp || kEnt);         // log p of K indices
    constexpr bool kSlice = (MODE == kModeSliceStats);  // a vocabulary slice's partials
    constexpr bool kGather = (kLogpFwd || kSelGrad || kSlice);  // K indices
    // + sum of logits (label smoothing; the fused mode runs only for few rows,
    // where the extra add costs nothing)
    constexpr bool kSumx =
        (MODE == kModeCeSmooth || MODE == kModeCeCapSmooth || MODE == kModeFused);
    constexpr int kH = kEnt ? kHMoment : (kSumx ? kHSum : kHNone);  // what h holds
    // a logit as the softmax sees it (soft-capped in the capped modes)
    const auto capped = [&](float x) { return kCap ? p.softcap * tanhf(x * p.inv_cap) : x; };
    const CapConsts capk = cap_consts(p.softcap, p.inv_cap, p.c);
    constexpr int kPasses = (MODE == kModeFused) ? 2 : 1;

    extern __shared__ __align__(128) uint8_t dyn_smem[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + (kRingAlign - 1)) & ~uintptr_t(kRingAlign - 1));
    __shared__ uint64_t full_bar[kStages];
    __shared__ uint64_t empty_bar[kStages];
    __shared__ float red_m[NCW], red_s[NCW], red_h[NCW];
    __shared__ int32_t red_i[NCW];
    __shared__ float s_xt[KMAX];
    __shared__ float s_dt[KMAX];       // kModeLogpGrad: gradient at each gathered column
    __shared__ float s_G, s_lp0;       // kModeLogpGrad: sum of upstream, log p of index 0
    __shared__ float s_gH, s_H;        // kModeLogpEntGrad: dL/dH and H of the row
    __shared__ int32_t s_tg[KMAX];
    __shared__ float bc_m, bc_s, bc_h, bc_logp;
    __shared__ uint64_t xbar;                   // cluster of CTAs per row: partials landed
    __shared__ uint64_t xt_bar;                 // statistics: s_xt written
    __shared__ __align__(16) float4 xchg[kMaxClusterCtas];  // every CTA's (m, s, h) partial

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t unit = blockIdx.x;
    const int64_t r = unit / p.splits;
    const int split = static_cast<int>(unit - r * p.splits);
    const int64_t V = p.vocab;
    const T *row = static_cast<const T *>(p.logits) + r * p.row_stride;
    T *drow = kGrad ? static_cast<T *>(p.dlogits) + r * p.d_stride : nullptr;

    // statistics over a vocabulary split: the row's CTAs form a cluster and
    // send their (m, s, h) partials through distributed shared memory to the
    // first CTA (to every CTA in the fused mode, which needs log p for its
    // gradient slice)
    const bool exchange = (kStats && p.splits > 1);
    // the mbarriers first: their setup overlaps the row selection's loads
    // (a skipped row leaves them unused)
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
        if (exchange)
            mbar_init(&xbar, 1);
        if (kStats)
            mbar_init(&xt_bar, 1);
        fence_barrier_init();
    }
    __syncthreads();  // the mbarriers exist before anyone uses them

    // this unit's body: 16-byte vectors [v0, v1) of the row, in chunks
    // (chunk i of a two-pass unit is chunk i mod nchunks of the body)
    const RowGeom g = row_geom<T>(row, V);
    const int64_t v0 = p.splits == 1 ? 0 : g.nvec * split / p.splits;
    const int64_t v1 = p.splits == 1 ? g.nvec : g.nvec * (split + 1) / p.splits;
    const int64_t nchunks = (v1 - v0 + CV - 1) / CV;
    const int64_t total = nchunks * kPasses;
    const char *body = reinterpret_cast<const char *>(row + g.head) + v0 * 16;
    const int64_t body_bytes = (v1 - v0) * 16;
    // copy chunk i into its ring slot (the statistics pass of a two-pass
    // unit keeps its bytes in L2 for the gradient pass)
    const auto issue_chunk = [&](int64_t i, uint64_t keep, uint64_t stream) {
        const int slot = static_cast<int>(i % kStages);
        const int64_t off = (i % nchunks) * kChunkBytes;
        const int64_t left = body_bytes - off;
        const uint32_t bytes = static_cast<uint32_t>(left < kChunkBytes ? left : kChunkBytes);
        const bool first_of_two = (kPasses == 2 && i < nchunks);
        mbar_arrive_expect_tx(&full_bar[slot], bytes);
        bulk_load(ring + slot * kChunkBytes, body + off, bytes, &full_bar[slot],
                  first_of_two ? keep : stream);
    };
    // A row split over several CTAs (few rows: latency, not bandwidth, sets
    // the pace) starts streaming before its row selection is known: the
    // producer issues the ring's first copies at once, and if the row turns
    // out to be skipped it waits for them to land before the CTA exits.
    int64_t issued = 0;
    if (p.splits > 1 && warp == NCW && lane == 0) {
        const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
        for (; issued < total && issued < kStages; ++issued)
            issue_chunk(issued, keep, stream);
    }

    // ---- row selection, before any read of this row's logits
    int32_t tg[KMAX];
    int32_t y = -1;
    int state = 0;  // 0 live, 1 skipped (ignored label / masked row), 2 bad label / index
    if (kGather) {
        // (the mask and the indices are read together: one memory latency).
        // A vocabulary slice holds the global columns [vocab_offset,
        // vocab_offset + V): a target elsewhere is simply not here.
        const bool slice = p.vocab_total > 0;
        const int64_t range = slice ? p.vocab_total : V;
        bool any_bad = false;
        int64_t first = -1;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int64_t t = k < p.k ? p.targets[r * p.k + k] : -1;
            if (k == 0)
                first = t;
            any_bad |= k < p.k && (t < 0 || t >= range);
            const int64_t loc = slice ? t - p.vocab_offset : t;
            tg[k] = (k < p.k && t >= 0 && t < range && loc >= 0 && loc < V)
                        ? static_cast<int32_t>(loc)
                        : -1;
        }
        if ((p.row_mask != nullptr && p.row_mask[r] == 0) ||
            (slice && first == p.ignore_index)) {
            state = 1;
            any_bad = false;
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                tg[k] = -1;
        }
        // the forward NaNs just the bad (r, k); its gradient NaNs the row
        if (kSelGrad && any_bad)
            state = 2;
    } else {
        const int64_t lab = p.targets[r];
        if (lab == p.ignore_index)
            state = 1;
        else if (lab < 0 || lab >= V)
            state = 2;
        y = state == 0 ? static_cast<int32_t>(lab) : -1;
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            tg[k] = (k == 0) ? y : -1;
    }

    if (state != 0) {
        // (every CTA of a row's cluster takes this exit together: nothing is
        // exchanged for the row)
        const float fill = state == 1 ? 0.0f : __int_as_float(0x7fc00000);
        // the first slice's CTA writes the row's outputs
        const bool direct = split == 0;
        if (kLogpFwd) {
            if (direct && tid < p.k)
                p.logp_out[r * p.k + tid] = 0.0f;
            if (kEnt && direct && tid == 0)
                p.entropy_out[r] = 0.0f;
        } else if (kSlice) {
            // a skipped row's partials: an empty state and no target logits
            float *part = p.slice_partials + r * (2 + p.k);
            if (direct && tid < 2 + p.k)
                part[tid] = tid == 0 ? kNegInf : 0.0f;
        } else if (kSelGrad) {
            if (tid == 0 && split == 0 && state == 2)
                report(p.dev_status, GBCE_DEV_BAD_INDEX);
            fill_row_slice<T>(drow, V, split, p.splits, fill);
        } else {
            if (tid == 0 && direct && state == 2)
                report(p.dev_status, GBCE_DEV_BAD_LABEL);
            if (tid == 0 && direct && !kCeGrad) {
                p.loss_rows[r] = fill;
                if (p.logp_out)
                    p.logp_out[r] = fill;
                if (p.lse_out)
                    p.lse_out[r] = fill;
            }
            if (kGrad)
                fill_row_slice<T>(drow, V, split, p.splits, fill);
        }
        // no copy may still be in flight when the CTA exits
        for (int64_t j = 0; j < issued; ++j)
            mbar_wait(&full_bar[j], 0);
        return;
    }

    if (exchange)
        cluster_arrive_relaxed();

    // ------------------------------------------------------------ producer
    if (warp == NCW) {
        if (lane == 0 && total > 0) {
            const uint64_t keep = policy_evict_last();
            const uint64_t stream = policy_evict_first();
            int64_t i = issued;  // (a split row's first copies are already on their way)
            bool ok = true;
            for (; i < total; ++i) {
                const int slot = static_cast<int>(i % kStages);
                if (i >= kStages &&
                    !mbar_wait(&empty_bar[slot], static_cast<uint32_t>((i / kStages - 1) & 1))) {
                    ok = false;
                    break;
                }
                issue_chunk(i, keep, stream);
            }
            if (!ok)
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            if (kStats && ok && total > kStages && p.prefetch_ahead > 0 &&
                r + p.prefetch_ahead < p.rows) {
                // the start of the row about to follow this CTA on its SM
                // (one CTA per row here), unless that row is skipped: its
                // first ring's worth of logits, so that its first copies
                // come from L2.  Taken once this CTA's last copy is issued
                // (a few chunks before its sweep ends), and only by the
                // statistics sweeps: the read+write gradient streams have no
                // bandwidth to spare for it.
                const int64_t r2 = r + p.prefetch_ahead;
                bool live = true;
                if (kGather)
                    live = p.row_mask == nullptr || p.row_mask[r2] != 0;
                else
                    live = p.targets[r2] != p.ignore_index;
                if (live) {
                    const T *row2 = static_cast<const T *>(p.logits) + r2 * p.row_stride;
                    const RowGeom g2 = row_geom<T>(row2, V);
                    const int64_t b2 = g2.nvec * 16;
                    const int64_t ring_bytes = static_cast<int64_t>(kStages) * kChunkBytes;
                    if (b2 > 0)
                        bulk_prefetch_l2(row2 + g2.head,
                                         static_cast<uint32_t>(b2 < ring_bytes ? b2 : ring_bytes));
                }
            }
            // no copy may still be in flight when the CTA exits
            for (int64_t j = (i > kStages ? i - kStages : 0); j < i; ++j)
                mbar_wait(&full_bar[j % kStages], static_cast<uint32_t>((j / kStages) & 1));
        }
        if (kStats && lane == 1) {
            // the target logits, for the finalize step: read by an idle
            // producer lane, so that no consumer waits on these dependent
            // loads before its sweep (all issued, then all stored)
            float xt[KMAX];
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                xt[k] = (k < p.k && tg[k] >= 0) ? E::load(row + tg[k]) : 0.0f;
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                if (k < p.k)
                    s_xt[k] = tg[k] >= 0 ? capped(xt[k]) : 0.0f;
            mbar_arrive(&xt_bar);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    // Per-row constants, computed while the producer already streams (no
    // use of a target index comes before this point, so the producer starts
    // as soon as the row selection is known -- at once for an unmasked
    // log-prob row).
    int32_t tv[KMAX];
    target_vectors<T, KMAX>(tg, g, tv);
    if (kSelGrad) {
        // gathered column t: (1/T)(-g_t expm1(log p_t) - (G - g_t) exp(log p_t)),
        // g_t the upstream of every k that gathers t; every other column j:
        // -(G/T) exp((x_j - x_{t0})/T + log p_{t0}).  The entropy term adds
        // -(gH/T) p_j (log p_j + H) to every column (0 where p_j = 0).
        // G - g_t is summed from the other indices' upstream (a difference of
        // G and g_t would keep a small upstream only to a large one's
        // rounding), and each sum of at most K upstream values is taken in
        // fp64 (in fp32 a sum that cancels keeps only its terms' rounding).
        if (tid < p.k) {
            const float *gr = p.grad_out + r * p.k;
            double G2 = 0.0, gt2 = 0.0, go2 = 0.0;
            int32_t mine = -1;
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                if (k == tid)
                    mine = tg[k];
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                if (k < p.k) {
                    const double gk = gr[k];
                    G2 += gk;
                    if (tg[k] == mine)
                        gt2 += gk;
                    else
                        go2 += gk;
                }
            // divided by T before they meet the probabilities: a product that
            // lands in the subnormals keeps its one rounding instead of having
            // it scaled by 1/T
            const float G = static_cast<float>(G2);
            const float gtT = static_cast<float>(gt2 / p.T), goT = static_cast<float>(go2 / p.T);
            const float lp = p.saved_logp[r * p.k + tid];
            float dt = fmaf(-gtT, expm1f(lp), -goT * expf(lp));
            float gH = 0.0f, H = 0.0f;
            if (kEntGrad) {
                gH = p.grad_entropy[r];
                H = p.saved_entropy[r];
                const float pt = expf(lp);
                if (pt > 0.0f)
                    dt -= (gH / p.T) * pt * (lp + H);
            }
            s_dt[tid] = dt;
            if (tid == 0) {
                s_G = G;
                s_lp0 = lp;
                s_gH = gH;
                s_H = H;
                s_xt[0] = p.target_logit != nullptr ? p.target_logit[r] : E::load(row + mine);
            }
        }
    }
    if (kStats) {
        // target columns, for the finalize step (read after the merge's
        // barrier; the producer warp reads their logits)
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            if (tid == k)
                s_tg[k] = tg[k];
    }
    if (kSelGrad)
        named_sync(1, NC);  // the gradient constants before the sweep uses them

    const float c = p.c;
    int64_t seq = 0;  // chunk sequence number across passes (slot, parity)
    bool alive = true;
    float logp = 0.0f, xy = 0.0f;
    float fm = kNegInf, fs = 0.0f;  // fused: the non-target columns' (max, sum)

    if (kStats) {
        OnlineStats<kEnt, kSumx> st;
        // each thread's next target vector; a warp none of whose threads
        // holds one skips even the cursor test (warp-uniform branch)
        int32_t nt = next_target_vector<KMAX>(tv, v0, v1, tid, NC, -1);
        const bool wcheck = __any_sync(0xffffffffu, nt != INT32_MAX);
        float mraw = capped_sweep_start();  // soft-capped sweep: the raw max behind st.m
        bool in_range = true;               // (unused here: no gradient pass follows)
        if (split == 0)
            for (int64_t e = tid; e < g.head; e += NC) {
                const float x = capped(E::load(row + e));
                st.add1(is_target<KMAX>(tg, static_cast<int32_t>(e)) ? kNegInf : x, c);
                st.sumx_add(x);
            }
        if (split == p.splits - 1)
            for (int64_t e = g.tail0 + tid; e < V; e += NC) {
                const float x = capped(E::load(row + e));
                st.add1(is_target<KMAX>(tg, static_cast<int32_t>(e)) ? kNegInf : x, c);
                st.sumx_add(x);
            }
        for (int64_t i = 0; i < nchunks; ++i, ++seq) {
            const int slot = static_cast<int>(seq % kStages);
            if (alive && !mbar_wait(&full_bar[slot], static_cast<uint32_t>((seq / kStages) & 1))) {
                alive = false;
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            }
            if (alive) {
                const uint4 *chunk = reinterpret_cast<const uint4 *>(ring + slot * kChunkBytes);
                const int64_t nv = (v1 - v0 - i * CV) < CV ? (v1 - v0 - i * CV) : CV;
                const int32_t vb0 = static_cast<int32_t>(v0 + i * CV);  // body vector of chunk[0]
                const int32_t col0 = static_cast<int32_t>(g.head);
                if (kCap && nv == CV) {
                    uint4 raw[PER_THREAD];
#pragma unroll
                    for (int u = 0; u < PER_THREAD; ++u)
                        raw[u] = chunk[tid + u * NC];
                    stats_capped_chunk<T, KMAX, PER_THREAD>(st, mraw, in_range, raw, vb0, col0,
                                                           nt, tg, tv, v0, v1, tid, NC, wcheck,
                                                           c, capk);
                } else if (kCap) {
                    for (int v = tid; v < nv; v += NC) {
                        const int32_t vb = vb0 + v;
                        if (wcheck && nt == vb) {
                            stats_capped_target<T, KMAX>(st, chunk[v], col0 + vb * VEC, tg, c,
                                                         capk);
                            nt = next_target_vector<KMAX>(tv, v0, v1, tid, NC, vb);
                            continue;
                        }
                        const uint4 one[1] = {chunk[v]};
                        const float own = raw_vmax<T, 1>(one);
                        stats_capped<T, 1>(st, mraw, in_range, one, own, own, c, capk);
                    }
                } else if (nv == CV) {
                    uint4 raw[PER_THREAD];
#pragma unroll
                    for (int u = 0; u < PER_THREAD; ++u)
                        raw[u] = chunk[tid + u * NC];
#pragma unroll
                    for (int u = 0; u + 1 < PER_THREAD; u += 2)
                        stats_two<T, KMAX, false>(st, raw[u], raw[u + 1], vb0 + tid + u * NC,
                                                  vb0 + tid + (u + 1) * NC, col0, nt, tg, c, tv,
                                                  v0, v1, tid, NC, wcheck);
                    if (PER_THREAD & 1)
                        stats_one<T, KMAX>(st, raw[PER_THREAD - 1],
                                           vb0 + tid + (PER_THREAD - 1) * NC, col0, nt, tg, c, tv,
                                           v0, v1, tid, NC, wcheck);
                } else {
                    for (int v = tid; v < nv; v += NC)
                        stats_one<T, KMAX>(st, chunk[v], vb0 + v, col0, nt, tg, c, tv, v0, v1,
                                           tid, NC, wcheck);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty_bar[slot]);
        }

        // the target logits have landed (long since: the loads were issued
        // when the sweep began); every reader of s_xt comes after this
        if (alive && !mbar_wait(&xt_bar, 0)) {
            alive = false;
            report(p.dev_status, GBCE_DEV_TIMEOUT);
        }

        // CTA-wide merge of the per-thread (max, sum[, h]) in a fixed order;
        // h is the entropy moment (kEnt) or the sum of logits (kSumx)
        float m = st.m, s = st.sum(), h = kEnt ? st.hsum() : (kSumx ? st.xsum() : 0.0f);
        if (kEnt && alive && isnan(h) && !isnan(s))
            h = rescan_entropy_moment<T, KMAX>(row, g, V, v0, v1, split == 0,
                                               split == p.splits - 1, tg, c, st.nmc, tid, NC);
        warp_merge_state<kH>(m, s, h, c, st.residual(c));
        if (lane == 0) {
            red_m[warp] = m;
            red_s[warp] = s;
            red_h[warp] = h;
        }
        named_sync(1, NC);
        if (warp == 0) {
            m = lane < NCW ? red_m[lane] : kNegInf;
            s = lane < NCW ? red_s[lane] : 0.0f;
            h = lane < NCW ? red_h[lane] : 0.0f;
            warp_merge_state<kH>(m, s, h, c);
            if (exchange)
                cluster_wait();  // every peer's mbarriers exist
            if (exchange && lane == 0) {
                const uint32_t C = static_cast<uint32_t>(p.splits);
                const bool all = (MODE == kModeFused);
                if (all || split == 0)
                    mbar_arrive_expect_tx(&xbar, C * static_cast<uint32_t>(sizeof(float4)));
                const uint32_t slot = smem_addr(&xchg[split]);
                const uint32_t bar = smem_addr(&xbar);
                const float4 part = make_float4(m, s, h, 0.0f);
                for (uint32_t t = 0; t < (all ? C : 1u); ++t)
                    st_async_v4(map_to_rank(slot, t), part, map_to_rank(bar, t));
            }
        }
        // a statistics-only CTA of a split row is done once its partial is sent
        if (exchange && MODE != kModeFused && split != 0)
            return;
        if (exchange && warp == 0) {
            // the partials of every slice, merged in slice order
            if (!mbar_wait_cluster(&xbar, 0)) {
                alive = false;
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            }
            m = kNegInf;
            s = 0.0f;
            h = 0.0f;
            for (int t = 0; t < p.splits; ++t) {
                const float4 part = xchg[t];
                merge_state<kH>(m, s, h, part.x, part.y, part.z, c);
            }
        }
        if (warp == 0 && lane == 0) {
            if (kLogpFwd) {
                bc_m = m;
                bc_s = s;
                bc_h = h;
            } else if (kSlice) {
                p.slice_partials[r * (2 + p.k)] = m;
                p.slice_partials[r * (2 + p.k) + 1] = s;
            } else {
                xy = s_xt[0];
                logp = finalize_logp(m, s, xy, p.T);
                if (split == 0) {
                    p.loss_rows[r] = ce_row_loss(logp, xy, h, p.T, p.ls_eps, p.dft, V);
                    if (p.logp_out)
                        p.logp_out[r] = logp;
                    if (p.lse_out)
                        p.lse_out[r] = xy / p.T - logp;
                }
                bc_logp = logp;
                bc_m = m;
                bc_s = s;
            }
        }
        if (kSlice && tid < p.k)  // the logits of the targets this slice holds
            p.slice_partials[r * (2 + p.k) + 2 + tid] = s_tg[tid] >= 0 ? s_xt[tid] : 0.0f;
        if (kLogpFwd) {
            named_sync(1, NC);
            // the last warp finalizes the entropy while warp 0 writes the
            // log-probs; a row that needs the second look gets it from that
            // warp alone, so no other warp waits for it
            if (kEnt && warp == NCW - 1) {
                bool rescan = false;
                float H = 0.0f;
                if (lane == 0)
                    H = entropy_with_targets<KMAX>(bc_m, bc_s, bc_h, s_tg, s_xt,
                                                   static_cast<int>(p.k), c, p.T, rescan);
                if (__shfl_sync(0xffffffffu, rescan, 0)) {
                    // confident in a column other than the first index: the
                    // entropy again, around that column, from the whole row
                    const RowGeom gr = row_geom<T>(row, V);
                    float M;
                    int32_t d;
                    row_argmax<T, 1>(row, gr, V, lane, nullptr, nullptr, M, d);
                    H = entropy_around<T, 1>(row, gr, V, d, M, c, p.T, lane, nullptr, nullptr,
                                             nullptr);
                }
                if (lane == 0)
                    p.entropy_out[r] = H;
            }
            if (tid < p.k) {
                float out;
                if (s_tg[tid] < 0) {
                    out = __int_as_float(0x7fc00000);
                    report(p.dev_status, GBCE_DEV_BAD_INDEX);
                } else {
                    out = logp_with_targets<KMAX>(bc_m, bc_s, s_tg, s_xt, static_cast<int>(p.k),
                                                  tid, c, p.T);
                }
                p.logp_out[r * p.k + tid] = out;
            }
        }
        if (MODE == kModeFused) {
            named_sync(1, NC);
            logp = bc_logp;
            xy = s_xt[0];
            fm = bc_m;
            fs = bc_s;
        }
    }

    if (kSelGrad) {
        GradConsts gk =
            kEntGrad ? grad_consts_ent(s_xt[0], c, s_lp0, -fmaf(s_gH, s_H, s_G) / p.T, -s_gH / p.T)
                     : grad_consts(s_xt[0], c, s_lp0, -s_G / p.T);
        // the exponents' reference: the first gathered column, or for a row
        // far below its max, the max itself (rebase_grad_consts)
        float xref = s_xt[0], lref2 = s_lp0 * kLog2e;
        if (s_lp0 < kRebaseLogp && (!slice_row(p) || p.row_state != nullptr)) {
            float M, S;
            if (slice_row(p)) {  // a vocabulary slice: the combine's whole-row state
                M = p.row_state[2 * r];
                S = p.row_state[2 * r + 1];
            } else {
                row_max_sum<T, NCW, false>(row, g, V, tid, c, 0.0f, 0.0f, red_m, red_s, M, S);
            }
            rebase_grad_consts(gk, M, S);
            if (S > 0.0f && isfinite(M)) {
                xref = M;
                lref2 = -log2f(S);
            }
        }
        const auto elem = [&](float x) {
            return kEntGrad ? grad_scalar_ent(x, gk) : grad_scalar(x, gk);
        };
        float dtv[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
            dtv[k] = s_dt[k];
        // With the entropy term, a row confident in a column d outside the
        // gathered set (p_t0 < 1/2 and H < 1/16) gets d's element from a
        // whole-row pass first: there the term needs H + log p_d, which the
        // per-element formula would take as a difference of nearly equal
        // numbers.  Its value then patches d like a gathered column.
        int32_t dcol = -1, dvec = -1;
        float dval = 0.0f;
        if (kEntGrad && s_gH != 0.0f && s_H < 0.0625f && s_lp0 < -0.69314718f) {
            float M;
            int32_t d;
            row_argmax<T, NCW>(row, g, V, tid, red_m, red_i, M, d);
            bool gathered = false;
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                gathered |= (tg[k] == d);
            if (!gathered && d < V) {
                const float Q = entropy_gap<T, NCW>(row, g, V, d, M, xref, lref2, c,
                                                    1.0f / p.T, tid, red_m);
                const float pd = ex2(fmaf(M - xref, c, lref2));
                dval = pd * (-(s_G / p.T) - (s_gH / p.T) * Q);
                dcol = d;
                dvec = (d >= g.head && d < g.tail0) ? static_cast<int32_t>((d - g.head) / VEC) : -1;
            }
        }
        const auto at_target = [&](int32_t col, float dflt) {
            float v = col == dcol ? dval : dflt;
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                v = (tg[k] == col) ? dtv[k] : v;
            return v;
        };
        constexpr int32_t kNoLabel = 0x7fffffff;
        if (split == 0)
            for (int64_t e = tid; e < g.head; e += NC)
                E::store(drow + e, at_target(static_cast<int32_t>(e), elem(E::load(row + e))));
        if (split == p.splits - 1)
            for (int64_t e = g.tail0 + tid; e < V; e += NC)
                E::store(drow + e, at_target(static_cast<int32_t>(e), elem(E::load(row + e))));
        for (int64_t i = 0; i < nchunks; ++i, ++seq) {
            const int slot = static_cast<int>(seq % kStages);
            if (alive && !mbar_wait(&full_bar[slot], static_cast<uint32_t>((seq / kStages) & 1))) {
                alive = false;
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            }
            if (alive) {
                const uint4 *chunk = reinterpret_cast<const uint4 *>(ring + slot * kChunkBytes);
                const int64_t nv = (v1 - v0 - i * CV) < CV ? (v1 - v0 - i * CV) : CV;
                const int64_t vbase = v0 + i * CV;
                T *dbase = drow + g.head + vbase * VEC;
                for (int v = tid; v < nv; v += NC) {
                    const uint4 raw = chunk[v];
                    const int32_t vb = static_cast<int32_t>(vbase + v);
                    if (!vector_has_target<KMAX>(tv, vb) && vb != dvec && p.vec_store) {
                        st_cs_v4(dbase + v * VEC,
                                 GradVec<T>::template run<kEntGrad>(raw, kNoLabel, gk));
                        continue;
                    }
                    float d[VEC];
                    GradVec<T>::template run_unpacked<kEntGrad>(raw, kNoLabel, gk, d);
                    const int32_t col0v = static_cast<int32_t>(g.head) + vb * VEC;
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        d[e] = at_target(col0v + e, d[e]);
                    if (p.vec_store) {
                        st_cs_v4(dbase + v * VEC, E::pack(d));
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            E::store(dbase + v * VEC + e, d[e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty_bar[slot]);
        }
    } else if (kGrad) {
        if (kCeGrad) {
            logp = p.saved_logp[r];
            xy = capped(E::load(row + y));
        }
        GradConsts gk =
            grad_consts_ce(xy, c, logp, upstream_grad(p, r), p.T, p.ls_eps, p.dft, V);
        // the exponents' reference moved to the row's max (rebase_grad_consts):
        // the fused call has the row's state at hand; ce_bwd reads it again for
        // a row far below its max
        if (MODE == kModeFused) {
            float M, S;
            row_state_with_target(fm, fs, xy, c, M, S);
            rebase_grad_consts(gk, M, S);
        } else if (kCeGrad && logp < kRebaseLogp) {
            float M, S;
            row_max_sum<T, NCW, kCap>(row, g, V, tid, c, p.softcap, p.inv_cap, red_m, red_s, M,
                                      S);
            rebase_grad_consts(gk, M, S);
        }
        if (kCap) {
            // soft-capped: element j is (its plain value on z = cap tanh(x / cap))
            // times the chain factor 1 - tanh^2(x / cap) (tanh_chain)
            const auto elem = [&](float x, bool is_y) {
                const float u = x * p.inv_cap;
                float unscale;
                const float chain = tanh_chain(u, unscale);
                const float z = p.softcap * tanhf(u);
                const float d = is_y ? gk.dy : fmaf(gk.gs, ex2(fmaf(z + gk.nxy, gk.c, gk.kb)), gk.c0);
                return (d * chain) * unscale;
            };
            if (split == 0)
                for (int64_t e = tid; e < g.head; e += NC)
                    E::store(drow + e, elem(E::load(row + e), e == y));
            if (split == p.splits - 1)
                for (int64_t e = g.tail0 + tid; e < V; e += NC)
                    E::store(drow + e, elem(E::load(row + e), e == y));
            for (int64_t i = 0; i < nchunks; ++i, ++seq) {
                const int slot = static_cast<int>(seq % kStages);
                if (alive &&
                    !mbar_wait(&full_bar[slot], static_cast<uint32_t>((seq / kStages) & 1))) {
                    alive = false;
                    report(p.dev_status, GBCE_DEV_TIMEOUT);
                }
                if (alive) {
                    const uint4 *chunk = reinterpret_cast<const uint4 *>(ring + slot * kChunkBytes);
                    const int64_t nv = (v1 - v0 - i * CV) < CV ? (v1 - v0 - i * CV) : CV;
                    const int64_t vbase = v0 + i * CV;
                    const int64_t col_base = g.head + vbase * VEC;
                    T *dbase = drow + col_base;
                    if (nv == CV && p.vec_store) {
                        grad_capped_chunk<T, PER_THREAD>(
                            chunk, dbase, static_cast<int32_t>(y - col_base), tid, NC, false, gk,
                            capk);
                    } else {
                        for (int v = tid; v < nv; v += NC) {
                            const int64_t yoff = y - (col_base + v * VEC);
                            if (p.vec_store && (yoff < 0 || yoff >= VEC)) {
                                st_cs_v4(dbase + v * VEC, grad_capped<T>(chunk[v], gk, capk));
                                continue;
                            }
                            float f[VEC];
                            E::unpack(chunk[v], f);
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                f[e] = elem(f[e], col_base + v * VEC + e == y);
                            if (p.vec_store) {
                                st_cs_v4(dbase + v * VEC, E::pack(f));
                            } else {
#pragma unroll
                                for (int e = 0; e < VEC; ++e)
                                    E::store(dbase + v * VEC + e, f[e]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty_bar[slot]);
            }
            return;
        }
        if (split == 0)
            for (int64_t e = tid; e < g.head; e += NC)
                E::store(drow + e, e == y ? gk.dy : grad_scalar(E::load(row + e), gk));
        if (split == p.splits - 1)
            for (int64_t e = g.tail0 + tid; e < V; e += NC)
                E::store(drow + e, e == y ? gk.dy : grad_scalar(E::load(row + e), gk));
        for (int64_t i = 0; i < nchunks; ++i, ++seq) {
            const int slot = static_cast<int>(seq % kStages);
            if (alive && !mbar_wait(&full_bar[slot], static_cast<uint32_t>((seq / kStages) & 1))) {
                alive = false;
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            }
            if (alive) {
                const uint4 *chunk = reinterpret_cast<const uint4 *>(ring + slot * kChunkBytes);
                const int64_t nv = (v1 - v0 - i * CV) < CV ? (v1 - v0 - i * CV) : CV;
                const int64_t vbase = v0 + i * CV;
                const int32_t ybase = y - static_cast<int32_t>(g.head + vbase * VEC);
                T *dbase = drow + g.head + vbase * VEC;
                if (nv == CV && p.vec_store) {
                    uint4 raw[PER_THREAD];
#pragma unroll
                    for (int u = 0; u < PER_THREAD; ++u)
                        raw[u] = chunk[tid + u * NC];
#pragma unroll
                    for (int u = 0; u < PER_THREAD; ++u) {
                        const int v = tid + u * NC;
                        st_cs_v4(dbase + v * VEC, GradVec<T>::run(raw[u], ybase - v * VEC, gk));
                    }
                } else if (p.vec_store) {
                    for (int v = tid; v < nv; v += NC)
                        st_cs_v4(dbase + v * VEC, GradVec<T>::run(chunk[v], ybase - v * VEC, gk));
                } else {
                    for (int v = tid; v < nv; v += NC) {
                        float d[VEC];
                        GradVec<T>::run_unpacked(chunk[v], ybase - v * VEC, gk, d);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            E::store(dbase + v * VEC + e, d[e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty_bar[slot]);
        }
    }
}

// The opt-in to more than 48 KB of dynamic shared memory is an attribute of
// the function in each device's context: set it once per device.
template <typename Kernel>
static cudaError_t ensure_smem_attr(Kernel kernel, int bytes, std::atomic<uint64_t> &done)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit) != 0)
        return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess)
        done.fetch_or(bit, std::memory_order_relaxed);
    return err;
}

// Launch configuration of `units` row-kernel CTAs in clusters of C.
struct ClusterLaunch {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    ClusterLaunch(int64_t units, int C, cudaStream_t stream)
    {
        cfg.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
        cfg.blockDim = dim3(kRowThreads, 1, 1);
        cfg.dynamicSmemBytes = kDynSmemBytes;
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(C);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
};

// The largest cluster size C <= want for which `rows` clusters of this
// kernel are all resident at once (one wave; a cluster must fit in one GPC,
// so this is below rows x C <= the CTA slots), 1 if none is.  The occupancy
// query runs once per device and size.
template <typename Kernel>
static int one_wave_cluster_size(Kernel kernel, int want, int64_t rows,
                                 std::atomic<int> (&cache)[64][kMaxClusterCtas + 1])
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return want;
    for (int C = want; C > 1; --C) {
        int n = cache[dev][C].load(std::memory_order_relaxed);
        if (n == 0) {
            ClusterLaunch l(static_cast<int64_t>(C) * rows, C, nullptr);
            if (cudaOccupancyMaxActiveClusters(&n, kernel, &l.cfg) != cudaSuccess || n < 1) {
                (void)cudaGetLastError();
                return want;  // no answer: keep the requested split
            }
            cache[dev][C].store(n, std::memory_order_relaxed);
        }
        if (n >= rows)
            return C;
    }
    return 1;
}

// One CTA per work unit.  Split statistics (p.splits > 1 in a statistics or
// fused mode) run each row's slices as one thread-block cluster, whose CTAs
// swap partials through distributed shared memory; the cluster shrinks from
// p.splits until every row's cluster is resident at once.
template <typename T, int MODE, int KMAX>
static cudaError_t launch_row_kernel(const RowParams &p, cudaStream_t stream)
{
    static std::atomic<uint64_t> attr_done{0};
    static std::atomic<int> max_clusters[64][kMaxClusterCtas + 1] = {};
    auto kernel = row_kernel<T, MODE, KMAX>;
    cudaError_t err = ensure_smem_attr(kernel, kDynSmemBytes, attr_done);
    if (err != cudaSuccess)
        return err;
    constexpr bool kStatsMode = !(MODE == kModeGrad || MODE == kModeGradCap ||
                                  MODE == kModeLogpGrad || MODE == kModeLogpEntGrad);
    RowParams q = p;
    if (kStatsMode && q.splits > 1)
        q.splits = one_wave_cluster_size(kernel, q.splits, q.rows, max_clusters);
    const int64_t units = q.rows * q.splits;
    q.prefetch_ahead = 0;
    if (kStatsMode && q.splits == 1) {
        // CTAs resident at once: a launch of more than that many rows warms
        // each next row in L2 from the CTA it follows
        static std::atomic<int> per_sm{0};
        int n = per_sm.load(std::memory_order_relaxed);
        if (n == 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kRowThreads,
                                                              kDynSmemBytes) == cudaSuccess)
                per_sm.store(n, std::memory_order_relaxed);
            else
                (void)cudaGetLastError();  // no prefetch; the launch itself decides
        }
        const int64_t resident = static_cast<int64_t>(n) * device_sm_count();
        if (resident > 0 && units > resident)
            q.prefetch_ahead = resident;
    }
    if (!kStatsMode || q.splits == 1) {
        kernel<<<static_cast<unsigned>(units), kRowThreads, kDynSmemBytes, stream>>>(q);
        note_launches(1);
        return cudaGetLastError();
    }
    ClusterLaunch l(units, q.splits, stream);
    err = cudaLaunchKernelEx(&l.cfg, kernel, q);
    note_launches(1);
    return err;
}

template <typename T>
cudaError_t launch_rows_dispatch(const RowParams &p, int mode, cudaStream_t stream);

template <typename T>
cudaError_t launch_rows(const RowParams &p, int mode, cudaStream_t stream)
{
    if (p.rows == 0)
        return cudaSuccess;
    return launch_rows_dispatch<T>(p, mode, stream);
}

// One CTA per work unit (clusters of them for split statistics): every call
// that the persistent kernel does not take.
template <typename T>
cudaError_t launch_rows_per_unit(const RowParams &p, int mode, cudaStream_t stream)
{
    switch (mode) {
    case kModeLogp:
        if (p.k <= 1)
            return launch_row_kernel<T, kModeLogp, 1>(p, stream);
        if (p.k <= 4)
            return launch_row_kernel<T, kModeLogp, 4>(p, stream);
        return launch_row_kernel<T, kModeLogp, GBCE_MAX_K>(p, stream);
    case kModeLogpEnt:
        if (p.k <= 1)
            return launch_row_kernel<T, kModeLogpEnt, 1>(p, stream);
        if (p.k <= 4)
            return launch_row_kernel<T, kModeLogpEnt, 4>(p, stream);
        return launch_row_kernel<T, kModeLogpEnt, GBCE_MAX_K>(p, stream);
    case kModeCe:
        return launch_row_kernel<T, kModeCe, 1>(p, stream);
    case kModeCeSmooth:
        return launch_row_kernel<T, kModeCeSmooth, 1>(p, stream);
    case kModeCeCap:
        return launch_row_kernel<T, kModeCeCap, 1>(p, stream);
    case kModeCeCapSmooth:
        return launch_row_kernel<T, kModeCeCapSmooth, 1>(p, stream);
    case kModeSliceStats:
        if (p.k <= 1)
            return launch_row_kernel<T, kModeSliceStats, 1>(p, stream);
        if (p.k <= 4)
            return launch_row_kernel<T, kModeSliceStats, 4>(p, stream);
        return launch_row_kernel<T, kModeSliceStats, GBCE_MAX_K>(p, stream);
    case kModeGradCap:
        return launch_row_kernel<T, kModeGradCap, 1>(p, stream);
    case kModeGrad:
        return launch_row_kernel<T, kModeGrad, 1>(p, stream);
    case kModeFused:
        return launch_row_kernel<T, kModeFused, 1>(p, stream);
    case kModeLogpGrad:
        if (p.k <= 1)
            return launch_row_kernel<T, kModeLogpGrad, 1>(p, stream);
        if (p.k <= 4)
            return launch_row_kernel<T, kModeLogpGrad, 4>(p, stream);
        return launch_row_kernel<T, kModeLogpGrad, GBCE_MAX_K>(p, stream);
    case kModeLogpEntGrad:
        if (p.k <= 1)
            return launch_row_kernel<T, kModeLogpEntGrad, 1>(p, stream);
        if (p.k <= 4)
            return launch_row_kernel<T, kModeLogpEntGrad, 4>(p, stream);
        return launch_row_kernel<T, kModeLogpEntGrad, GBCE_MAX_K>(p, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace gbce
