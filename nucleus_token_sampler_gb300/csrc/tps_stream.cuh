// tps_stream.cuh -- the streaming sampler: one persistent CTA per SM, whole rows streamed through a
// ring of bulk-copied chunks.  Used when the batch has enough rows to fill the GPU.
//
// Thread 0 keeps the ring full: each free stage receives the next 32 KB chunk of the CTA's next
// row (`cp.async.bulk` into this CTA's shared memory, completed on that stage's mbarrier), so the
// HBM stream never waits for the arithmetic.  All 256 threads consume chunks in order.  While a row
// streams, they keep its running maximum and list every token that min-p, measured against the
// running maximum, does not already reject; the running maximum only grows, so the list is a
// superset of the row's survivors.  At the end of the row the list is filtered exactly against the
// true maximum and resolved (top-k, top-p, race) while the ring already holds the next row's
// chunks.  Rows without min-p, or whose list overflows, take the general path, which reads the row
// again from global memory (it was just streamed, so mostly from L2).
#pragma once

#include "tps_common.cuh"

namespace tps {

constexpr int kMaxStages = 16;

struct StreamState {
    uint64_t full[kMaxStages];  // one mbarrier per ring stage
    float cmax[2][kWarps];      // per-warp chunk maxima, double-buffered by chunk parity
    float xmax[kWarps];         // per-warp maxima of the ragged elements
    uint32_t dead;              // a bounded wait gave up: the CTA stops streaming
};

// Geometry of one row: aligned interior in 16-byte vectors plus a ragged head and tail.
struct RowGeom {
    const unsigned char* rowp;
    uintptr_t a0;      // 16-byte-aligned start of the interior
    int64_t n16;       // interior vectors
    int nhead, ntail;  // ragged elements before / after the interior
    int nchunks;       // interior chunks
};

template <int ES>
__device__ __forceinline__ RowGeom row_geom(const Args& a, int64_t row, uint32_t chunk_bytes)
{
    RowGeom g;
    g.rowp = static_cast<const unsigned char*>(a.logits) + row * a.ld * ES;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(g.rowp), g1 = g0 + (uintptr_t)a.V * ES;
    uintptr_t a0 = (g0 + 15) & ~(uintptr_t)15, a1 = g1 & ~(uintptr_t)15;
    if (a1 <= a0) {
        g.a0 = g1;
        g.n16 = 0;
        g.nhead = (int)a.V;
        g.ntail = 0;
    } else {
        g.a0 = a0;
        g.n16 = (int64_t)(a1 - a0) / 16;
        g.nhead = (int)((a0 - g0) / ES);
        g.ntail = (int)((g1 - a1) / ES);
    }
    g.nchunks = (int)((g.n16 * 16 + chunk_bytes - 1) / chunk_bytes);
    return g;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1) stream_rows_kernel(const Args a, int nstage, uint32_t chunk_bytes)
{
    using E = Elem<TIn>;
    constexpr int ES = E::kBytes;
    extern __shared__ __align__(128) unsigned char dsmem[];
    unsigned char* ring = dsmem;
    Shared& s = *reinterpret_cast<Shared*>(dsmem + (size_t)nstage * chunk_bytes);
    StreamState& st = *reinterpret_cast<StreamState*>(reinterpret_cast<unsigned char*>(&s) + sizeof(Shared));
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t B = a.B;
    const int64_t first = blockIdx.x, stride = gridDim.x;
    const int chunk_vecs = (int)(chunk_bytes / 16);

    // ---- producer state (thread 0 only): the next chunk to issue
    int64_t p_row = first;
    int p_chunk = 0;
    RowGeom p_geom;
    uint64_t issued = 0;
    if (tid == 0) {
        for (int i = 0; i < nstage; ++i) mbar_init(&st.full[i], 1);
        st.dead = 0;
        if (p_row < B) p_geom = row_geom<ES>(a, p_row, chunk_bytes);
    }
    __syncthreads();
    // Issue the next chunk into its stage; false when the CTA has no chunk left.
    auto issue_one = [&]() -> bool {
        while (p_row < B && p_chunk >= p_geom.nchunks) {
            p_row += stride;
            p_chunk = 0;
            if (p_row < B) p_geom = row_geom<ES>(a, p_row, chunk_bytes);
        }
        if (p_row >= B || st.dead) return false;
        const int stage = (int)(issued % (uint64_t)nstage);
        const uint64_t off = (uint64_t)p_chunk * chunk_bytes;
        const uint32_t bytes = (uint32_t)min((uint64_t)chunk_bytes, (uint64_t)p_geom.n16 * 16 - off);
        fence_proxy_async();
        mbar_arrive_expect_tx(&st.full[stage], bytes);
        bulk_g2s(ring + (size_t)stage * chunk_bytes, reinterpret_cast<const unsigned char*>(p_geom.a0) + off, bytes,
                 &st.full[stage]);
        ++p_chunk;
        ++issued;
        return true;
    };
    if (tid == 0)
        for (int i = 0; i < nstage; ++i)
            if (!issue_one()) break;

    uint64_t consumed = 0;
    // per-row parameters, prefetched one row ahead
    auto load_params = [&](int64_t row, float& T, float& P, float& MP, int32_t& K, uint64_t& seed) {
        if (row < B) {
            T = a.temperature[row];
            P = a.top_p[row];
            MP = a.min_p[row];
            K = a.top_k[row];
            seed = a.seed[row];
        }
    };
    float nT = 0.f, nP = 0.f, nMP = 0.f;
    int32_t nK = 0;
    uint64_t nSeed = 0;
    load_params(first, nT, nP, nMP, nK, nSeed);

    for (int64_t row = first; row < B; row += stride) {
        const float T = nT, P = nP, MP = nMP;
        const int32_t K = nK;
        const uint64_t seed = nSeed;
        load_params(row + stride, nT, nP, nMP, nK, nSeed);
        const RowGeom g = row_geom<ES>(a, row, chunk_bytes);
        const bool params_ok = isfinite(T) && isfinite(P) && isfinite(MP);
        const bool sampling = params_ok && T > 0.f;
        const float minp = (MP > 0.f) ? fminf(MP, 1.f) : 0.f;
        const bool listing = sampling && minp > 0.f;
        const float lt_hi = listing ? make_ctx(0.f, T, minp).L_hi * T * (1.f + 1e-5f) : 0.f;

        // ragged head/tail: loads issued now, used after the last chunk
        const int nx = g.nhead + g.ntail;
        float xv = -INFINITY;
        int32_t xidx = 0;
        if (tid < nx) {
            xidx = (tid < g.nhead) ? tid : (int32_t)(a.V - g.ntail + (tid - g.nhead));
            xv = E::load1(g.rowp, xidx);
        }
        if (tid == 0) s.ncand = 0;
        // (the barrier at the end of the first chunk, or below, orders this reset)

        float runmax = -INFINITY;  // maximum over the chunks finished so far (same in every thread)
        float thr = INFINITY;      // list tokens with z > thr
        auto set_thr = [&]() {
            thr = (listing && runmax > -INFINITY && runmax < INFINITY) ? list_threshold(runmax, lt_hi) : INFINITY;
            if (isnan(thr)) thr = INFINITY;
        };
        auto list_token = [&](float z, int32_t i) {
            const uint32_t slot = atomicAdd(&s.ncand, 1u);
            if (slot < (uint32_t)kCand) {
                s.ckey[slot] = fkey(z);
                s.cidx[slot] = (uint32_t)i;
            }
        };
        bool dead = st.dead != 0;  // after a timeout nothing more is streamed
        for (int c = 0; c < g.nchunks && !dead; ++c) {
            const int stage = (int)(consumed % (uint64_t)nstage);
            const uint32_t parity = (uint32_t)((consumed / (uint64_t)nstage) & 1u);
            const uint64_t off = (uint64_t)c * chunk_bytes;
            const int nv = (int)min((uint64_t)chunk_vecs, (uint64_t)g.n16 - off / 16);
            const uint4* cv = reinterpret_cast<const uint4*>(ring + (size_t)stage * chunk_bytes);
            const int32_t e0 = g.nhead + (int32_t)(off / ES);
            uint32_t to = mbar_wait_bounded(&st.full[stage], parity, kWaitLimitNs) ? 0u : 1u;
            if (__syncthreads_or(to)) {
                dead = true;
                break;
            }
            auto nolist = [](float, int32_t) {};
            float cm;
            if (c == 0) {
                // first chunk: its own maximum sets the first listing threshold
                cm = warp_max_nan(scan_max_list<TIn, false>(cv, nv, e0, INFINITY, nolist));
                if (lane == 0) st.cmax[1][warp] = cm;
                __syncthreads();
                float m0 = st.cmax[1][0];
#pragma unroll
                for (int w = 1; w < kWarps; ++w) m0 = fmax_nan(m0, st.cmax[1][w]);
                runmax = m0;
                set_thr();
                if (listing) (void)scan_max_list<TIn, false>(cv, nv, e0, thr, list_token);
                cm = m0;
            } else {
                cm = warp_max_nan(scan_max_list<TIn, false>(cv, nv, e0, thr, list_token));
            }
            const int par = c & 1;
            if (lane == 0) st.cmax[par][warp] = cm;
            __syncthreads();  // the stage is free; every warp's chunk maximum is visible
            if (tid == 0) (void)issue_one();
            float m = runmax;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) m = fmax_nan(m, st.cmax[par][w]);
            if (!(m == runmax)) {
                runmax = m;
                set_thr();
            }
            ++consumed;
        }

        // ---- the ragged elements, then the row's exact maximum
        float xm = (tid < nx) ? xv : -INFINITY;
        xm = warp_max_nan(xm);
        if (lane == 0) st.xmax[warp] = xm;
        if (tid < nx) {
            s.xz[tid] = xv;
            s.xi[tid] = xidx;
        }
        if (tid == 0) s.nx = nx;
        __syncthreads();
        float zmax = runmax;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) zmax = fmax_nan(zmax, st.xmax[w]);
        // the ragged elements are listed against the exact maximum (a threshold at least as low as
        // any running one would give, so the list stays a superset of the survivors)
        if (tid < nx && listing && zmax > -INFINITY && zmax < INFINITY &&
            xv > minp_threshold(make_ctx(zmax, T, minp)))
            list_token(xv, xidx);
        const bool cta_dead = __syncthreads_or(dead || st.dead) != 0;
        if (cta_dead && tid == 0) st.dead = 1;

        int32_t status = kRowOk;
        if (cta_dead) status = kRowTimeout;
        else if (isnan(zmax) || zmax == INFINITY) status = kRowNan;
        else if (!params_ok) status = kRowBadParam;
        else if (zmax == -INFINITY) status = kRowAllMasked;

        float* prow = a.out_probs ? a.out_probs + row * a.V : nullptr;
        GlobalRow<TIn> src;
        src.vec = reinterpret_cast<const uint4*>(g.a0);
        src.nvec = (int)g.n16;
        src.elem0 = g.nhead;

        if (status != kRowOk) {
            if (prow)
                for (int64_t i = tid; i < a.V; i += kThreads) prow[i] = 0.f;
            if (tid == 0) write_row(a, row, -1, status, __uint_as_float(0x7FC00000u), 0);
            __syncthreads();
            continue;
        }
        if (T <= 0.f) {
            // greedy: lowest index of the maximum ("Implement batched top-p sampling with temperature",
            // 'A strong answer': temperature 0 means greedy, ties to the lowest index)
            uint32_t mi = 0xFFFFFFFFu;
            src.for_each(s, [&](float z, int32_t i) {
                if (z == zmax) mi = min(mi, (uint32_t)i);
            });
            mi = block_min_u32(mi, s);
            if (prow)
                for (int64_t i = tid; i < a.V; i += kThreads) prow[i] = ((uint32_t)i == mi) ? 1.f : 0.f;
            if (tid == 0) write_row(a, row, (int32_t)mi, kRowOk, zmax, 1);
            __syncthreads();
            continue;
        }

        const RowCtx r = make_ctx(zmax, T, minp);
        const float zc = minp_threshold(r);
        const bool topk_on = (K > 0) && ((int64_t)K < a.V);
        RaceCtx rc;
        rc.k0 = (uint32_t)seed;
        rc.k1 = (uint32_t)(seed >> 32);
        rc.row = (uint32_t)row;
        rc.s_lo = (uint32_t)a.step;
        rc.s_hi = (uint32_t)(a.step >> 32);

        const uint32_t nlisted = s.ncand;
        RowResult res;
        if (listing && nlisted <= (uint32_t)kCand && thr > -INFINITY) {
            // every survivor is on the list: filter it exactly against the true maximum
            __syncthreads();
            if (tid == 0) s.ncand = 0;
            __syncthreads();
            if ((uint32_t)tid < nlisted) {
                const uint32_t key = s.ckey[tid];
                const float z = key_to_float(key);
                if (z > zc && minp_ok(r, z, dist(r, z))) {
                    const uint32_t slot = atomicAdd(&s.ncand, 1u);
                    s.u.cd.sbuf[slot] = sb_make(key, s.cidx[tid]);
                }
            }
            __syncthreads();
            res = resolve_candidates(s, r, rc, s.ncand, topk_on, K, P);
            if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
        } else {
            SoloTopo topo;
            res = general_path(topo, s, src, r, zc, topk_on, K, P, rc, prow);
        }
        if (tid == 0) write_row(a, row, res.token, kRowOk, key_to_float(res.key_cut), (int32_t)res.nk);
        __syncthreads();  // the row's shared state may be reused
    }

    // Copies still in flight (only after a timeout) must land before the shared memory is released.
    if (tid == 0 && st.dead) {
        for (uint64_t g2 = consumed; g2 < issued; ++g2)
            (void)mbar_wait_bounded(&st.full[g2 % (uint64_t)nstage], (uint32_t)((g2 / (uint64_t)nstage) & 1u),
                                    kWaitLimitNs);
    }
}

}  // namespace tps
