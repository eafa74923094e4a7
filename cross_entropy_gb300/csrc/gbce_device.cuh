// Device helpers for the sm_103a kernels: mbarrier / bulk-copy (TMA) PTX with
// bounded waits, cache policies, and the online (max, sum) state of a row
// sweep.  Nothing here allocates; nothing here waits without a limit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbce {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

// ---------------------------------------------------------------- PTX: smem

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization may start while the kernel before it in the stream
// still runs.  grid_dependency_wait blocks the calling thread until that
// kernel has completed and its memory writes are visible (at once when the
// kernel was launched without the attribute).  launch_dependents lets the
// kernel after this one start before this one ends.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Same, with acquire at cluster scope: for barriers whose transactions are
// stores from other CTAs of the cluster.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, giving up after
// ~2 s or 2^26 polls (each try_wait itself suspends for a bounded time).
// Returns false on timeout.  Every pipeline wait in this library goes
// through here, so no kernel can spin forever on a copy that never lands.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it < (1u << 26); ++it) {
#ifdef GBCE_WAIT_SLEEP_NS  // build option: back off between polls
        __nanosleep(GBCE_WAIT_SLEEP_NS);
#endif
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0 && global_timer_ns() - t0 > 2000000000ull)
            break;
    }
    return false;
}

// Bounded wait for a barrier completed by peer CTAs' st.async stores.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it < (1u << 26); ++it) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if ((it & 63u) == 0 && global_timer_ns() - t0 > 2000000000ull)
            break;
    }
    return false;
}

// L2 eviction-priority policies for bulk copies.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared (TMA engine), completion signalled on `bar`
// as transaction bytes.  src, dst and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Bring `bytes` of global memory at `src` into L2 (no destination, no
// completion to wait for); src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Named barrier over the first `threads` threads of the CTA (warp multiple).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------ PTX: thread-block clusters

// The cluster barrier in two halves.  Every thread of every CTA arrives
// once, right after its CTA's mbarriers are initialised (whose
// fence.mbarrier_init makes them visible to the cluster); the relaxed arrive
// orders nothing else.  A thread that is about to store into a peer's shared
// memory first waits, which returns once every non-exited thread of the
// cluster has arrived -- so no store reaches a peer before the peer's
// mbarriers exist.  The CTAs of a cluster are co-scheduled and arrive at
// their start, so the wait does not depend on any data.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_address, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_address), "r"(rank));
    return r;
}

// Store four floats into a peer CTA's shared memory (16-byte aligned);
// completion is counted as 16 transaction bytes on the peer's mbarrier at
// `remote_bar`.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float4 v, uint32_t remote_bar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(remote_addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}

// ---------------------------------------------------------- PTX: global mem

__device__ __forceinline__ uint4 ld_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Streaming 16-byte store: the gradient is written once and not re-read.
__device__ __forceinline__ void st_cs_v4(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------- arithmetic

// 2^x on the SFU (relative error ~2^-22; results below 2^-126 flush to 0).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float softplus(float a)
{
    return fmaxf(a, 0.0f) + log1pf(expf(-fabsf(a)));
}

// ------------------------------------------------- packed fp32 (sm_100+)
// Two fp32 lanes per instruction: fma/add/mul.rn.f32x2 on a 64-bit register.

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// 1 / x to about 1 ulp (0 for +inf).
__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ soft-capping
//
// A soft-capped logit is cap * tanh(x / cap).  The few values that set a
// row's log p to full accuracy -- the row max and the target -- use CUDA's
// tanhf.  The bulk of a row goes through tanh_pair below, in packed pairs.
// Written as t = tanh(u), u = x / cap, the capped logit cap * t enters the
// softmax through the exponent t * (cap * log2(e) / T) + shift, so cap
// costs no extra multiply.

// Range of the series form: |u| < kCapSeriesBound.
constexpr float kCapSeriesBound = 0.55f;

// tanh(u) = u P(s), s = u^2, for |u| < kCapSeriesBound, with P(s) = 1 +
// s Q(s) and Q the cubic fitted to (tanh(u) / u - 1) / s on that range by
// weighted least squares in relative error (near-minimax): 3.7e-8 relative
// in exact arithmetic, about 1.5 ulp evaluated in fp32.  The form is odd in
// u: no abs and no sign fix-up.
constexpr float kTanhQ0 = -0.3333294657493646f, kTanhQ1 = 0.13320723563804557f,
                kTanhQ2 = -0.052671713622700365f, kTanhQ3 = 0.016437383467281172f;

// scale * P(s) by Horner in packed pairs, from the pre-scaled coefficients
// sq[k] = scale * kTanhQk and s0 = scale (4 fused multiply-adds).
__device__ __forceinline__ float2 tanh_poly_pair(float2 s, const float (&sq)[4], float s0)
{
    float2 h = make_float2(sq[3], sq[3]);
    h = ffma2(h, s, make_float2(sq[2], sq[2]));
    h = ffma2(h, s, make_float2(sq[1], sq[1]));
    h = ffma2(h, s, make_float2(sq[0], sq[0]));
    return ffma2(h, s, make_float2(s0, s0));
}

__device__ __forceinline__ float2 tanh_series_pair(float2 u)
{
    const float q[4] = {kTanhQ0, kTanhQ1, kTanhQ2, kTanhQ3};
    return fmul2(u, tanh_poly_pair(fmul2(u, u), q, 1.0f));
}

// tanh(u) for any u, one lane at a time: the series below kCapSeriesBound,
// else t = 1 - 2 r with r = 1 / (e + 1), e = e^{2|u|} (t >= 0.5 there, so
// nothing cancels; e = +inf gives t = 1).
__device__ __forceinline__ float tanh_lane(float u)
{
    const float a = fabsf(u);
    if (a < kCapSeriesBound)
        return tanh_series_pair(make_float2(u, u)).x;
    const float e = ex2(2.0f * 1.4426950408889634f * a);
    const float r = rcp_approx(e + 1.0f);
    return copysignf(fmaf(-2.0f, r, 1.0f), u);
}

// The soft-cap's chain factor 1 - tanh^2(u) = sech^2(u), to a few ulp
// relative for every u: (2 h / (1 + h^2))^2 with h = e^{-|u|}, a sum and a
// quotient of positive numbers (1 - t^2 from a rounded t loses every digit
// once t rounds to 1, from |u| of about 9).  Past |u| = 20 the factor
// (below 2^-55) would soon leave fp32's normal range: it comes back times
// 2^64, with *unscale = 2^-64 for the caller to apply to its final product,
// so that a gradient element down in the subnormals is rounded once.  The
// factor is 0 for |u| = inf, NaN for a NaN u.
__device__ __forceinline__ float tanh_chain(float u, float &unscale)
{
    const float a = fabsf(u);
    const bool far = a > 20.0f;
    const float h = expf(-a) * (far ? 0x1p32f : 1.0f);
    const float w = far ? 0.0f : h * h;  // far out, 1 + e^{-2|u|} rounds to 1
    const float q = __fdiv_rn(2.0f * h, 1.0f + w);
    unscale = far ? 0x1p-64f : 1.0f;
    return q * q;
}

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float fmin3(float a, float b, float c)
{
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Exact max / min of two packed bf16 pairs (a NaN operand yields the other one).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Max of v over the warp's active lanes, in one warp-wide reduction; a NaN
// lane is ignored unless every lane is NaN.
__device__ __forceinline__ float warp_max_active(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, %2;" : "=f"(r) : "f"(v), "r"(__activemask()));
    return r;
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Round a pair to bf16 (nearest even) and pack it, .x in the low half.
__device__ __forceinline__ uint32_t float2_to_bf16x2(float2 v)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
}

// Element access for the two logit types.
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[4])
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static __forceinline__ float load(const float *p) { return __ldg(p); }
    __device__ static __forceinline__ void store(float *p, float v) { *p = v; }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[8])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ static __forceinline__ float load(const __nv_bfloat16 *p)
    {
        return __bfloat162float(__ldg(p));
    }
    __device__ static __forceinline__ void store(__nv_bfloat16 *p, float v)
    {
        *p = __float2bfloat16_rn(v);
    }
};

// Online (max, sum) over a stream of logits, in the exp2 domain:
//   m = max x_j,   s = sum_j 2^{(x_j - m) c},   c = log2(e) / T,
// so that s = sum_j exp((x_j - m) / T).  Excluded columns are fed as -inf.
// The sum is kept in two packed pairs (four independent accumulators).
template <bool ENT, bool SUMX = false>
struct OnlineStats {
    static constexpr bool kSumx = SUMX;
    float m = kNegInf;
    float nmc = __builtin_huge_valf();  // -m * c, the shift added to every x * c
    float2 sa = make_float2(0.0f, 0.0f);
    float2 sb = make_float2(0.0f, 0.0f);
    // ENT: sums of 2^z * z, z = (x - m) c <= 0 (the entropy's first moment)
    float2 ha = make_float2(0.0f, 0.0f);
    float2 hb = make_float2(0.0f, 0.0f);
    // SUMX: plain sums of the raw logits, every column including targets
    float2 xa = make_float2(0.0f, 0.0f);
    float2 xb = make_float2(0.0f, 0.0f);

    // SUMX: add raw logits that the exp sums do not see as themselves
    // (target columns, masked to -inf there; vectors that are all -inf).
    __device__ __forceinline__ void sumx_add(float x)
    {
        if (SUMX)
            xa.x += x;
    }

    // New running maximum `vmax` for the values about to be added; returns
    // false when there is nothing to add (all of them are -inf).
    __device__ __forceinline__ bool raise_to(float vmax, float c)
    {
        if (vmax > m) {
            // every z so far was x c + nmc: moving the sums to the new shift
            // multiplies them by 2^(nmc' - nmc), a difference of the two
            // rounded shifts (exact when they are within a factor of two), so
            // all terms keep sharing one rounding of the shift (finish)
            const float nmc_new = -vmax * c;
            const float d = nmc_new - nmc;
            const float f = ex2(d);
            const float2 ff = make_float2(f, f);
            if (ENT && m != kNegInf) {
                // every z drops by -d: sum 2^z z -> f (sum 2^z z + d sum 2^z)
                const float2 dd = make_float2(d, d);
                ha = fmul2(ffma2(sa, dd, ha), ff);
                hb = fmul2(ffma2(sb, dd, hb), ff);
            }
            sa = fmul2(sa, ff);
            sb = fmul2(sb, ff);
            m = vmax;
            nmc = nmc_new;
        }
        return vmax != kNegInf;
    }

    // z with -inf raised to a finite value far below the ex2 range, so that a
    // -inf logit (2^z = 0) adds 0 to h instead of 0 * -inf; a NaN stays NaN.
    __device__ static __forceinline__ float zfin(float z) { return fmaxf(z, -0x1p100f); }

    // Add 2^{x c - m c} for the four values of two packed pairs.  The h terms
    // skip zfin (one instruction per element on the hot path): a -inf logit
    // here turns h into NaN while the sum stays finite, and the kernel then
    // rescans that thread's columns with zfin (rescan_entropy_moment).
    __device__ __forceinline__ void add_pairs(float2 p, float2 q, float c)
    {
        const float2 cc = make_float2(c, c), kk = make_float2(nmc, nmc);
        const float2 zp = ffma2(p, cc, kk), zq = ffma2(q, cc, kk);
        const float2 ep = make_float2(ex2(zp.x), ex2(zp.y));
        const float2 eq = make_float2(ex2(zq.x), ex2(zq.y));
        sa = fadd2(sa, ep);
        sb = fadd2(sb, eq);
        if (SUMX) {
            xa = fadd2(xa, p);
            xb = fadd2(xb, q);
        }
        if (ENT) {
            ha = ffma2(ep, zp, ha);
            hb = ffma2(eq, zq, hb);
        }
    }

    // Add 2^z for four precomputed exponents z = x c - m c in two pairs.
    __device__ __forceinline__ void add_exponent_pairs(float2 zp, float2 zq)
    {
        sa = fadd2(sa, make_float2(ex2(zp.x), ex2(zp.y)));
        sb = fadd2(sb, make_float2(ex2(zq.x), ex2(zq.y)));
    }

    // SUMX: add two pairs of logits to the plain sums.
    __device__ __forceinline__ void sumx_pairs(float2 p, float2 q)
    {
        if (SUMX) {
            xa = fadd2(xa, p);
            xb = fadd2(xb, q);
        }
    }

    // Fold N unpacked values (masked columns already -inf).
    template <int N>
    __device__ __forceinline__ void add(const float (&f)[N], float vmax, float c)
    {
        if (!raise_to(vmax, c))
            return;
        float a = 0.0f, b = 0.0f, ah = 0.0f, bh = 0.0f;
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float za = fmaf(f[i], c, nmc);
            const float ea = ex2(za);
            a += ea;
            if (ENT)
                ah = fmaf(ea, zfin(za), ah);
            if (i + 1 < N) {
                const float zb = fmaf(f[i + 1], c, nmc);
                const float eb = ex2(zb);
                b += eb;
                if (ENT)
                    bh = fmaf(eb, zfin(zb), bh);
            }
        }
        sa.x += a;
        sb.x += b;
        if (ENT) {
            ha.x += ah;
            hb.x += bh;
        }
    }

    __device__ __forceinline__ void add1(float x, float c)
    {
        float f[1] = {x};
        add<1>(f, x, c);
    }

    // The thread's (max, sum) pair.
    __device__ __forceinline__ float sum() const
    {
        return __fadd_rn(__fadd_rn(sa.x, sa.y), __fadd_rn(sb.x, sb.y));
    }
    // Every exponent was evaluated as x c + nmc, nmc the rounded -m c, so
    // each carries the same r = m c + nmc (exact as one fma; |r| is at most
    // half an ulp of m c): the sums are 2^r times their values relative to
    // m.  warp_merge_state takes r out as it moves each lane to the warp's
    // max.  Left in, a row whose logits are large (|m| / T in the hundreds)
    // would carry ~2^-24 |m c| of error in every probability.
    __device__ __forceinline__ float residual(float c) const
    {
        return (m == kNegInf || !(m == m)) ? 0.0f : fmaf(m, c, nmc);
    }
    // ENT: the thread's sum of 2^z z.
    __device__ __forceinline__ float hsum() const
    {
        return __fadd_rn(__fadd_rn(ha.x, ha.y), __fadd_rn(hb.x, hb.y));
    }
    // SUMX: the thread's sum of raw logits.
    __device__ __forceinline__ float xsum() const
    {
        return __fadd_rn(__fadd_rn(xa.x, xa.y), __fadd_rn(xb.x, xb.y));
    }
};

using OnlineMaxSum = OnlineStats<false>;

// Merge two (max, sum) partial states with the same scale c.  Exactly
// commutative (no fused multiply-add): merging the slices of a row in slice
// order, or two partials in either order, gives the same bits.
__device__ __forceinline__ void merge_max_sum(float &m, float &s, float m2, float s2, float c)
{
    const float M = fmaxf(m, m2);
    if (M == kNegInf) {
        m = M;
        s = 0.0f;
        return;
    }
    s = __fadd_rn(__fmul_rn(s, ex2((m - M) * c)), __fmul_rn(s2, ex2((m2 - M) * c)));
    m = M;
}

// merge_max_sum for states that also carry h = sum 2^z z (z = (x - m) c):
// moving a part from its max m_i to M shifts its z by d_i = (m_i - M) c, so
// h_i -> 2^{d_i} (h_i + d_i s_i).  Exactly commutative like merge_max_sum.
__device__ __forceinline__ void merge_max_sum_h(float &m, float &s, float &h, float m2, float s2,
                                                float h2, float c)
{
    const float M = fmaxf(m, m2);
    if (M == kNegInf) {
        m = M;
        s = 0.0f;
        h = 0.0f;
        return;
    }
    const auto part = [&](float mi, float si, float hi, float &sv, float &hv) {
        if (mi == kNegInf) {
            sv = 0.0f;
            hv = 0.0f;
            return;
        }
        const float d = __fmul_rn(__fsub_rn(mi, M), c);
        const float f = ex2(d);
        sv = __fmul_rn(si, f);
        hv = __fmul_rn(__fadd_rn(hi, __fmul_rn(d, si)), f);
    };
    float sa, ha, sb, hb;
    part(m, s, h, sa, ha);
    part(m2, s2, h2, sb, hb);
    s = __fadd_rn(sa, sb);
    h = __fadd_rn(ha, hb);
    m = M;
}

// What the third accumulator h of a row state (m, s, h) holds: nothing, the
// entropy moment sum 2^z z (rescaled with the max), or a plain sum (of raw
// logits, for label smoothing).
enum StateH : int { kHNone = 0, kHMoment = 1, kHSum = 2 };

// Merge two row states with the same scale c; exactly commutative.
template <int HK>
__device__ __forceinline__ void merge_state(float &m, float &s, float &h, float m2, float s2,
                                            float h2, float c)
{
    if (HK == kHMoment) {
        merge_max_sum_h(m, s, h, m2, s2, h2, c);
    } else {
        merge_max_sum(m, s, m2, s2, c);
        if (HK == kHSum)
            h = __fadd_rn(h, h2);
    }
}

// Sum over the 32 lanes of a warp by a butterfly of rounded adds: each add
// is commutative, so every lane ends with the same bits, in a fixed order.
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Merge the (m, s[, h]) states of the 32 lanes of a warp (all active) into
// one, on every lane: the warp's max in one reduction, each lane's sum (and
// moment: h -> 2^d (h + d s), d = (m - M) c - r) moved to it, then butterfly
// sums.  r is the lane's exponent residual (OnlineStats::residual; 0 for
// states that carry none).  A lane with m = -inf adds nothing; a NaN max is
// ignored by the max and turns the sums NaN.
template <int HK>
__device__ __forceinline__ void warp_merge_state(float &m, float &s, float &h, float c,
                                                 float r = 0.0f)
{
    float M;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(M) : "f"(m));
    float sv = 0.0f, hv = HK == kHSum ? h : 0.0f;
    if (M != kNegInf && m != kNegInf) {
        const float d = __fsub_rn(__fmul_rn(__fsub_rn(m, M), c), r);
        const float f = ex2(d);
        sv = __fmul_rn(s, f);
        if (HK == kHMoment)
            hv = __fmul_rn(__fadd_rn(h, __fmul_rn(d, s)), f);
    }
    m = M;
    s = warp_sum(sv);
    if (HK != kHNone)
        h = warp_sum(hv);
}

// log p_t from the others' (m, s) and the target logit, all in raw logit
// units: a = log s + (m - x_t) / T, log p = -softplus(a).  The margin
// (m - x_t) / T is one IEEE division of an exact (bf16) or once-rounded
// (fp32) difference, taken from the same values the sweep read, so log p
// is never positive.  s == 0 (no other column, V == 1) gives log p = 0.
__device__ __forceinline__ float finalize_logp(float m, float s, float xt, float T)
{
    if (!(s > 0.0f))
        return (s == 0.0f) ? 0.0f : __int_as_float(0x7fc00000);
    const float a = logf(s) + (m - xt) / T;
    return -softplus(a);
}

// Entropy -sum_j p_j log p_j of a row from the others' state (m, s, h) --
// every column but the reference column t, h = sum 2^z z in base-2 units --
// and x_t.  With a = log s + (m - x_t)/T (log p_t = -softplus(a)),
//   p_t = sigmoid(-a), 1 - p_t = sigmoid(a),
//   log sum_all e^{(x_j - m)/T} = log s + softplus(-a) =: L,
//   H = p_t softplus(a) + (1 - p_t) (L - ln2 h / s),
// a sum of non-negative terms: nothing cancels when t holds almost all of
// the mass (the confident rows), and 1 - p_t never rounds to 0 there.
// Past a = -80, 1 - p_t and softplus(a) both equal e^a to a relative e^a
// and fall below fp32's normal range, while H = e^a (1 + L - mean) may not:
// there e^a is carried times 2^64 (the square of e^{a/2} 2^32, both normal
// down to a = -174) and the product is scaled back in one rounding, so an
// entropy down to fp32's smallest subnormal keeps its value.
__device__ __forceinline__ float finalize_entropy(float m, float s, float h, float xt, float T)
{
    if (!(s > 0.0f))
        return (s == 0.0f) ? 0.0f : __int_as_float(0x7fc00000);
    const float ls = logf(s);
    const float a = ls + (m - xt) / T;
    const float mean_u = (h / s) * 0.69314718055994531f;  // <= 0
    if (a < -80.0f) {
        const float e2 = expf(0.5f * a) * 0x1p32f;
        return ((e2 * e2) * ((1.0f + ls - a) - mean_u)) * 0x1p-64f;
    }
    const float sp = softplus(a), spn = softplus(-a);
    const float pt = expf(-sp);  // e^{log p_t}
    const float q = -expm1f(-sp);
    const float ht = pt > 0.0f ? pt * sp : 0.0f;
    return fmaf(q, (ls + spn) - mean_u, ht);
}

}  // namespace gbce
