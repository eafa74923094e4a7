// Persistent fused cross-entropy forward + backward (sm_103a).
//
// One CTA per SM walks rows: row blockIdx.x first, then whichever row the
// next ticket names (gridDim.x + an atomic counter in the workspace, zeroed
// by the item-count kernel that runs before), so that CTAs that meet
// ignored rows or finish early take more rows and the last rows spread over
// every SM.  Its producer lane streams, without gaps, row r's statistics
// pass (bulk copies with L2 evict_last), row r's gradient pass (the same
// bytes again, now L2 hits), then the next row's statistics pass, ...
// through a ring of 48 KB stages, and hands each row's id to the consumer
// warps through a small queue in shared memory.  The consumer warps fold
// pass-1 chunks into the row's online (max, sum), finalize log p between
// the passes, and write dlogits from pass-2 chunks.
//
// Why one CTA per SM: a row must stay in L2 from its first read to its
// re-read, so the L2 footprint is (rows in flight) x (row bytes).  One row
// per SM (152 x 304 KB = 46 MB at vocab 152064 bf16) fits the 126 MB L2 next
// to the dlogits stream; two rows per SM, as one CTA per row at two CTAs per
// SM has, does not, and the gradient pass then re-reads part of each row
// from HBM.  Persistence keeps the ring full across row boundaries, so the
// one CTA never idles HBM while it merges a row's statistics.
//
// Sources, by title and section: the sum over the columns other than the
// target and loss = softplus(log s_others + m - x_y), "Fix softmax collapse
// in CE, GRPO, KL/JSD and softmax" (Liger-Kernel PR #1555), "Summary"; the
// -expm1(log p) target gradient, the unsloth-zoo #2080 commit quoted there,
// "Fix"; ignored rows skipped before any vocabulary read and g*softmax -
// g*onehot into a separate buffer, ms-swift PR #10353, "PR information".
#pragma once

#include "gbce_kernels.cuh"

namespace gbce {

// Shape of the persistent CTA (build options GBCE_PERSIST_* override it).
// Measured on GB300 at 8192 x 152064 bf16, consumer warps x chunk x stages:
// 8 x 32K x 4: 75%, 16 x 16K x 8: 80%, 16 x 64K x 2: 78%, 16 x 32K x 4: 86%,
// 20 x 40K x 4: 91.5%, 24 x 48K x 4: 94.8%, 28 x 28K x 4: 81% of measured
// HBM bandwidth -- more warps hide the exp chains' latency as long as each
// thread still gets four 16-byte vectors per chunk.  Later, with the
// one-barrier merge: 24 x 48K x 4 at 0.95-0.96 against 24 x 72K x 3 at 0.89
// and 24 x 24K x 8 at 0.90.
#ifndef GBCE_PERSIST_WARPS
#define GBCE_PERSIST_WARPS 24
#endif
#ifndef GBCE_PERSIST_CHUNK
#define GBCE_PERSIST_CHUNK 49152
#endif
#ifndef GBCE_PERSIST_STAGES
#define GBCE_PERSIST_STAGES 4
#endif
//
// The soft-capped kernel is bound by its FMA pipe rather than by HBM, and it
// runs two half-size CTAs per SM (12 consumer warps, a 4 x 24 KB ring each):
// one CTA's per-row merge then overlaps the other's sweep (1.18 -> 1.12 ms
// at 8192 rows).  The uncapped kernel loses with two rows per SM in flight
// (0.78 -> 0.90 ms): its gradient pass re-reads each row from L2, and twice
// the rows in flight crowd them out.
// L2 bytes the rows awaiting their gradient pass may take (see
// launch_persistent_fused_as).
constexpr int64_t kPersistL2Budget = int64_t(76) << 20;

template <bool CAP>
struct PersistShape {
    static constexpr int kWarps = CAP ? 12 : GBCE_PERSIST_WARPS;     // consumer warps
    static constexpr int kChunk = CAP ? 24576 : GBCE_PERSIST_CHUNK;  // bytes per ring stage
    static constexpr int kStages = CAP ? 4 : GBCE_PERSIST_STAGES;
    static constexpr int kCtasPerSm = CAP ? 2 : 1;
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kDynSmem = kStages * kChunk + kRingAlign;
};

// SMOOTH: label smoothing, which also needs each row's sum of logits.
// CAP: logit soft-capping, cap * tanh(x / cap) on every logit (and the
// chain factor 1 - tanh^2 in the gradient).
template <typename T, bool SMOOTH, bool CAP>
__global__ void __launch_bounds__(PersistShape<CAP>::kThreads, PersistShape<CAP>::kCtasPerSm)
    persistent_fused_kernel(const RowParams p)
{
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    using Shape = PersistShape<CAP>;
    constexpr int NCW = Shape::kWarps;
    constexpr int NC = NCW * 32;
    constexpr int S = Shape::kStages;
    constexpr int CHUNK = Shape::kChunk;
    constexpr int CV = CHUNK / 16;
    constexpr int PER_THREAD = CV / NC;
    static_assert(CV % NC == 0 && PER_THREAD % 2 == 0, "chunk must split evenly into pairs");
    static_assert(Shape::kThreads <= 1024, "at most 1024 threads per CTA");

    extern __shared__ __align__(128) uint8_t dyn_smem[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + (kRingAlign - 1)) & ~uintptr_t(kRingAlign - 1));
    __shared__ uint64_t full_bar[S];
    __shared__ uint64_t empty_bar[S];
    constexpr int Q = 4;  // row-id queue, producer -> consumers
    __shared__ uint64_t rq_full[Q], rq_empty[Q];
    __shared__ int32_t rq_row[Q];
    __shared__ int64_t rq_lab[Q];  // each handed-out row's label, read by the producer
    // per-warp partials of a row, double-buffered by the parity of the
    // consumers' live-row count: a warp that has merged one row can write
    // the next row's partials while a slower warp still reads this row's
    __shared__ float red_m[2][NCW], red_s[2][NCW], red_x[2][NCW];
    __shared__ int red_in[2][NCW];  // CAP: the warp's vectors all in the series range

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t V = p.vocab;
    const float c = p.c;
    const CapConsts capk = cap_consts(p.softcap, p.inv_cap, p.c);
    // a logit as the softmax sees it
    const auto capped = [&](float x) { return CAP ? p.softcap * tanhf(x * p.inv_cap) : x; };

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            mbar_init(&rq_full[q], 1);
            mbar_init(&rq_empty[q], NCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // launched as a programmatic dependent of the item count: the row
    // ticket, the row order and n_items are read only after it completes
    grid_dependency_wait();

    // ------------------------------------------------------------ producer
    if (warp == NCW) {
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();
            const uint64_t stream = policy_evict_first();
            uint32_t seq = 0;          // chunks issued
            uint32_t slot = 0, lap = 0;  // ring position of chunk seq, and its lap
            bool ok = true;
            // ticket t -> row: in the order the item count wrote when most
            // rows are ignored (live rows first, then the ignored ones, which
            // only write zeros and so even out the last rows' finishing
            // times), else row t
            const bool ordered = p.row_order != nullptr && *p.row_order_flag != 0;
            const auto row_of = [&](int64_t t) -> int64_t {
                return t >= p.rows ? p.rows : (ordered ? p.row_order[t] : t);
            };
            int64_t t = blockIdx.x;
            int64_t r = row_of(t);
            int64_t lab = r < p.rows ? p.targets[r] : 0;
            for (uint32_t qi = 0; ok; ++qi) {
                // hand row r (-1: no more rows) to the consumers
                const uint32_t qs = qi % Q;
                if (qi >= Q && !mbar_wait(&rq_empty[qs], ((qi / Q) - 1) & 1)) {
                    ok = false;
                    break;
                }
                rq_row[qs] = r < p.rows ? static_cast<int32_t>(r) : -1;
                rq_lab[qs] = lab;
                mbar_arrive(&rq_full[qs]);  // (release: the consumers see rq_row, rq_lab)
                if (r >= p.rows)
                    break;
                // the ticket for the row after this one, fetched while this
                // one streams (without a ticket counter: the static walk)
                const int64_t next_t =
                    p.row_ticket != nullptr
                        ? gridDim.x + static_cast<int64_t>(atomicAdd(p.row_ticket, 1))
                        : t + gridDim.x;
                const int64_t next = row_of(next_t);
                if (lab == p.ignore_index || lab < 0 || lab >= V) {
                    t = next_t;
                    r = next;
                    lab = r < p.rows ? p.targets[r] : 0;
                    continue;
                }
                // the next row's label, read while this row's gradient pass
                // streams (the ticket has long returned by then)
                int64_t next_lab = 0;
                const T *row = static_cast<const T *>(p.logits) + r * p.row_stride;
                const RowGeom g = row_geom<T>(row, V);
                const char *body = reinterpret_cast<const char *>(row + g.head);
                const int64_t bytes_total = g.nvec * 16;
                for (int pass = 0; pass < 2 && ok; ++pass) {
                    if (pass == 1 && next < p.rows)
                        next_lab = p.targets[next];
                    for (int64_t off = 0; off < bytes_total; off += CHUNK, ++seq) {
                        if (lap > 0 && !mbar_wait(&empty_bar[slot], (lap - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        const int64_t left = bytes_total - off;
                        const uint32_t bytes = static_cast<uint32_t>(left < CHUNK ? left : CHUNK);
                        mbar_arrive_expect_tx(&full_bar[slot], bytes);
                        bulk_load(ring + slot * CHUNK, body + off, bytes, &full_bar[slot],
                                  pass == 0 ? keep : stream);
                        if (++slot == S) {
                            slot = 0;
                            ++lap;
                        }
                    }
                }
                t = next_t;
                r = next;
                lab = next_lab;
            }
            if (!ok)
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            // no copy may still be in flight when the CTA exits
            for (uint32_t j = (seq > S ? seq - S : 0); j < seq; ++j)
                mbar_wait(&full_bar[j % S], (j / S) & 1);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    uint32_t slot = 0, lap = 0;  // ring position of the next chunk, and its lap
    bool alive = true;
    uint32_t live_rows = 0;  // rows merged so far (the partials' buffer parity)
    for (uint32_t qi = 0;; ++qi) {
        // the next row from the producer
        const uint32_t qs = qi % Q;
        if (!mbar_wait(&rq_full[qs], (qi / Q) & 1)) {
            report(p.dev_status, GBCE_DEV_TIMEOUT);
            break;
        }
        const int64_t r = rq_row[qs];
        const int64_t lab = rq_lab[qs];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&rq_empty[qs]);
        if (r < 0)
            break;
        const T *row = static_cast<const T *>(p.logits) + r * p.row_stride;
        T *drow = static_cast<T *>(p.dlogits) + r * p.d_stride;
        if (lab == p.ignore_index || lab < 0 || lab >= V) {
            const bool bad = lab != p.ignore_index;
            const float fill = bad ? __int_as_float(0x7fc00000) : 0.0f;
            if (tid == 0) {
                if (bad)
                    report(p.dev_status, GBCE_DEV_BAD_LABEL);
                p.loss_rows[r] = fill;
                if (p.logp_out)
                    p.logp_out[r] = fill;
                if (p.lse_out)
                    p.lse_out[r] = fill;
            }
            const RowGeom gd = row_geom<T>(drow, V);
            float f[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                f[e] = fill;
            const uint4 pat = E::pack(f);
            uint4 *body = reinterpret_cast<uint4 *>(drow + gd.head);
            for (int64_t v = tid; v < gd.nvec; v += NC)
                st_cs_v4(body + v, pat);
            for (int64_t e = tid; e < gd.head; e += NC)
                E::store(drow + e, fill);
            for (int64_t e = gd.tail0 + tid; e < V; e += NC)
                E::store(drow + e, fill);
            continue;
        }
        const int32_t y = static_cast<int32_t>(lab);
        const int32_t tg[1] = {y};
        const RowGeom g = row_geom<T>(row, V);
        int32_t tv[1];
        target_vectors<T, 1>(tg, g, tv);
        const int64_t nchunks = (g.nvec * 16 + CHUNK - 1) / CHUNK;
        const int32_t col0 = static_cast<int32_t>(g.head);
        // the label logit and the upstream gradient are read now (every thread,
        // one cached address each), so their latency hides under pass 1
        const float xy = capped(E::load(row + y));
        const float gup = upstream_grad(p, r);

        // pass 1: statistics
        OnlineStats<false, SMOOTH> st;
        int32_t nt = next_target_vector<1>(tv, 0, g.nvec, tid, NC, -1);
        const bool wcheck = __any_sync(0xffffffffu, nt != INT32_MAX);
        float mraw = capped_sweep_start();  // soft-capped sweep: the raw max behind st.m
        bool in_range = true;  // CAP: this thread's vectors all in the series range
        for (int64_t e = tid; e < g.head; e += NC) {
            const float x = capped(E::load(row + e));
            st.add1(e == y ? kNegInf : x, c);
            st.sumx_add(x);
        }
        for (int64_t e = g.tail0 + tid; e < V; e += NC) {
            const float x = capped(E::load(row + e));
            st.add1(e == y ? kNegInf : x, c);
            st.sumx_add(x);
        }
        for (int64_t i = 0; i < nchunks; ++i) {
            if (alive && !mbar_wait(&full_bar[slot], lap & 1)) {
                alive = false;
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            }
            if (alive) {
                const uint4 *chunk = reinterpret_cast<const uint4 *>(ring + slot * CHUNK);
                const int32_t vb0 = static_cast<int32_t>(i * CV);
                const int32_t nv = static_cast<int32_t>((g.nvec - i * CV) < CV ? (g.nvec - i * CV) : CV);
                if (CAP && nv == CV) {
                    uint4 raw[PER_THREAD];
#pragma unroll
                    for (int u = 0; u < PER_THREAD; ++u)
                        raw[u] = chunk[tid + u * NC];
                    stats_capped_chunk<T, 1, PER_THREAD>(st, mraw, in_range, raw, vb0, col0, nt,
                                                        tg, tv, 0, g.nvec, tid, NC, wcheck, c,
                                                        capk);
                } else if (CAP) {
                    for (int v = tid; v < nv; v += NC) {
                        const int32_t vb = vb0 + v;
                        if (wcheck && nt == vb) {
                            stats_capped_target<T, 1>(st, chunk[v], col0 + vb * VEC, tg, c, capk);
                            nt = next_target_vector<1>(tv, 0, g.nvec, tid, NC, vb);
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
                    for (int u = 0; u < PER_THREAD; u += 2)
                        stats_two<T, 1, true>(st, raw[u], raw[u + 1], vb0 + tid + u * NC,
                                              vb0 + tid + (u + 1) * NC, col0, nt, tg, c, tv, 0,
                                              g.nvec, tid, NC, wcheck);
                } else {
                    for (int v = tid; v < nv; v += NC)
                        stats_one<T, 1>(st, chunk[v], vb0 + v, col0, nt, tg, c, tv, 0, g.nvec,
                                        tid, NC, wcheck);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty_bar[slot]);
            if (++slot == S) {
                slot = 0;
                ++lap;
            }
        }

        // merge: each warp's state, one barrier, then every warp merges the
        // warps' states itself (no second barrier to broadcast log p)
        const int rb = static_cast<int>(live_rows++ & 1u);
        float m = st.m, s = st.sum(), sx = SMOOTH ? st.xsum() : 0.0f;
        warp_merge_state<SMOOTH ? kHSum : kHNone>(m, s, sx, c, st.residual(c));
        if (CAP)
            in_range = __all_sync(0xffffffffu, in_range);
        if (lane == 0) {
            red_m[rb][warp] = m;
            red_s[rb][warp] = s;
            red_x[rb][warp] = sx;
            if (CAP)
                red_in[rb][warp] = in_range;
        }
        named_sync(1, NC);
        m = lane < NCW ? red_m[rb][lane] : kNegInf;
        s = lane < NCW ? red_s[rb][lane] : 0.0f;
        sx = lane < NCW ? red_x[rb][lane] : 0.0f;
        if (CAP)
            in_range = __all_sync(0xffffffffu, lane < NCW ? red_in[rb][lane] != 0 : true);
        warp_merge_state<SMOOTH ? kHSum : kHNone>(m, s, sx, c);
        const float lp = finalize_logp(m, s, xy, p.T);
        if (tid == 0) {
            p.loss_rows[r] = ce_row_loss(lp, xy, sx, p.T, p.ls_eps, p.dft, V);
            if (p.logp_out)
                p.logp_out[r] = lp;
            if (p.lse_out)
                p.lse_out[r] = xy / p.T - lp;
        }
        GradConsts gk = grad_consts_ce(xy, c, lp, gup, p.T, p.ls_eps, p.dft, V);
        if (lp < kRebaseLogp) {
            // a row far below its max: the exponents' reference moves to the
            // max (rebase_grad_consts), whose state the merge just gave
            float M, S;
            row_state_with_target(m, s, xy, c, M, S);
            rebase_grad_consts(gk, M, S);
        }

        // pass 2: gradient
        // soft-capped element: its plain value on z = cap tanh(x / cap) times
        // the chain factor 1 - tanh^2(x / cap) (tanh_chain)
        const auto elem = [&](float x, bool is_y) {
            if (!CAP)
                return is_y ? gk.dy : grad_scalar(x, gk);
            const float u = x * p.inv_cap;
            float unscale;
            const float chain = tanh_chain(u, unscale);
            const float d =
                is_y ? gk.dy : fmaf(gk.gs, ex2(fmaf(tanhf(u), capk.capc, gk.kbx)), gk.c0);
            return (d * chain) * unscale;
        };
        for (int64_t e = tid; e < g.head; e += NC)
            E::store(drow + e, elem(E::load(row + e), e == y));
        for (int64_t e = g.tail0 + tid; e < V; e += NC)
            E::store(drow + e, elem(E::load(row + e), e == y));
        for (int64_t i = 0; i < nchunks; ++i) {
            if (alive && !mbar_wait(&full_bar[slot], lap & 1)) {
                alive = false;
                report(p.dev_status, GBCE_DEV_TIMEOUT);
            }
            if (alive) {
                const uint4 *chunk = reinterpret_cast<const uint4 *>(ring + slot * CHUNK);
                const int64_t vbase = i * CV;
                const int32_t nv = static_cast<int32_t>((g.nvec - vbase) < CV ? (g.nvec - vbase) : CV);
                const int32_t ybase = y - static_cast<int32_t>(g.head + vbase * VEC);
                T *dbase = drow + g.head + vbase * VEC;
                if (CAP && nv == CV && p.vec_store) {
                    grad_capped_chunk<T, PER_THREAD>(chunk, dbase, ybase, tid, NC, in_range, gk,
                                                     capk);
                } else if (CAP) {
                    for (int v = tid; v < nv; v += NC) {
                        const int32_t yoff = ybase - v * VEC;
                        if (p.vec_store && static_cast<uint32_t>(yoff) >= static_cast<uint32_t>(VEC)) {
                            st_cs_v4(dbase + v * VEC, grad_capped<T>(chunk[v], gk, capk));
                            continue;
                        }
                        float f[VEC];
                        E::unpack(chunk[v], f);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            f[e] = elem(f[e], e == yoff);
                        if (p.vec_store) {
                            st_cs_v4(dbase + v * VEC, E::pack(f));
                        } else {
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                E::store(dbase + v * VEC + e, f[e]);
                        }
                    }
                } else if (nv == CV && p.vec_store) {
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
            if (++slot == S) {
                slot = 0;
                ++lap;
            }
        }
    }
}

template <typename T, bool SMOOTH, bool CAP>
cudaError_t launch_persistent_fused_as(const RowParams &p, int sms, cudaStream_t stream)
{
    using Shape = PersistShape<CAP>;
    static std::atomic<uint64_t> attr_done{0};
    auto kernel = persistent_fused_kernel<T, SMOOTH, CAP>;
    cudaError_t err = ensure_smem_attr(kernel, Shape::kDynSmem, attr_done);
    if (err != cudaSuccess)
        return err;
    int64_t slots = static_cast<int64_t>(Shape::kCtasPerSm) * sms;
    if (!CAP) {
        // every CTA keeps one row in L2 from its first read to its re-read:
        // with long rows, fewer CTAs, so that those rows stay within about
        // 80 MB (fp32 rows of 152K columns: 131 CTAs, 0.43 -> 0.42 ms at
        // 2048 rows; 152 rows in flight, 92 MB, lose their re-read), but
        // never fewer than half the SMs (rows too long for L2 miss anyway)
        const int64_t row_bytes = p.vocab * static_cast<int64_t>(sizeof(T));
        const int64_t fit = kPersistL2Budget / (row_bytes > 0 ? row_bytes : 1);
        const int64_t floor = sms / 2 > 0 ? sms / 2 : 1;
        if (fit < slots)
            slots = fit > floor ? fit : floor;
    }
    const int grid = static_cast<int>(p.rows < slots ? p.rows : slots);
    // a programmatic dependent of the item count, which lets it start: the
    // CTAs' launch and prologue overlap the count
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Shape::kThreads);
    cfg.dynamicSmemBytes = Shape::kDynSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, p);
    note_launches(1);
    return err != cudaSuccess ? err : cudaGetLastError();
}

template <typename T>
cudaError_t launch_persistent_fused(const RowParams &p, int sms, cudaStream_t stream)
{
    if (p.softcap > 0.0f)
        return p.ls_eps != 0.0f ? launch_persistent_fused_as<T, true, true>(p, sms, stream)
                                : launch_persistent_fused_as<T, false, true>(p, sms, stream);
    return p.ls_eps != 0.0f ? launch_persistent_fused_as<T, true, false>(p, sms, stream)
                            : launch_persistent_fused_as<T, false, false>(p, sms, stream);
}

}  // namespace gbce
