// tps_stream.cuh -- the streaming sampler: one persistent CTA per SM, whole rows streamed through a
// ring of bulk-copied chunks.  Used when the batch has enough rows to fill the GPU.
//
// Warp-specialised pipeline.  One producer warp keeps the ring full: as soon as a stage is released
// it bulk-copies the next 64 KB chunk of the CTA's next row into it (`cp.async.bulk` into this
// CTA's shared memory, completed on the stage's "full" mbarrier).  Eight consumer warps scan the
// chunks and release each stage through its "empty" mbarrier -- no CTA-wide barrier per chunk, so
// the HBM stream never waits for the arithmetic.  While a row streams, every warp keeps its
// running maximum (also pooled across warps through an atomic maximum) and lists every token that
// min-p, measured against that running maximum, does not already reject; the running maximum only
// grows, so the list is a superset of the row's survivors.  At the end of the row the consumer
// warps meet once, filter the list exactly against the true maximum and resolve the row (top-k,
// top-p, race) while the producer already streams the next row.  Rows without min-p, or whose list
// overflows, take the general path, which re-reads the row from global memory (it was just
// streamed, so mostly from L2).
#pragma once

#include "tps_common.cuh"

namespace tps {

constexpr int kMaxStages = 8;
constexpr int kStreamThreads = kThreads + 32;  // consumer warps + one producer warp
constexpr int kStreamList = 2048;              // candidate list of one streamed row

struct StreamState {
    uint64_t full[kMaxStages];   // stage holds its chunk (arrive + transaction bytes)
    uint64_t empty[kMaxStages];  // every consumer warp is done with the stage
    float wmax[kWarps];          // per-warp maxima of the row (NaN-propagating)
    uint32_t runkey;             // order-preserving key of the pooled running maximum
    uint32_t dead;               // a bounded wait gave up: streaming stops
    uint32_t producer_done;      // the producer has left its loop
    uint32_t issued_lo;          // chunks issued (low 32 bits), valid once producer_done is set
    uint32_t lcount;             // tokens listed for the current row (may exceed kStreamList)
    uint32_t lkey[kStreamList];  // listed tokens: logit key and index
    uint32_t lidx[kStreamList];
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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <typename TIn>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_rows_kernel(const Args a, int nstage, uint32_t chunk_bytes)
{
    using E = Elem<TIn>;
    constexpr int ES = E::kBytes;
    extern __shared__ __align__(128) unsigned char dsmem[];
    unsigned char* ring = dsmem;
    Shared& s = *reinterpret_cast<Shared*>(dsmem + (size_t)nstage * chunk_bytes);
    StreamState& st = *reinterpret_cast<StreamState*>(reinterpret_cast<unsigned char*>(&s) + sizeof(Shared));
    volatile uint32_t* vdead = &st.dead;
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t B = a.B;
    const int64_t first = blockIdx.x, stride = gridDim.x;
    const uint32_t key_neg_inf = 0x007FFFFFu;  // fkey(-inf)

    if (tid == 0) {
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&st.full[i], 1);
            mbar_init(&st.empty[i], kWarps);
        }
        st.dead = 0;
        st.producer_done = 0;
        st.issued_lo = 0;
        st.runkey = key_neg_inf;
        st.lcount = 0;
    }
    __syncthreads();  // the only barrier the producer warp joins

    // ================= producer warp =================
    if (warp == kWarps) {
        if (lane == 0) {
            uint64_t g = 0;
            for (int64_t row = first; row < B && !*vdead; row += stride) {
                const RowGeom geo = row_geom<ES>(a, row, chunk_bytes);
                for (int c = 0; c < geo.nchunks; ++c, ++g) {
                    const int stage = (int)(g % (uint64_t)nstage);
                    if (g >= (uint64_t)nstage) {
                        const uint32_t ph = (uint32_t)(((g / (uint64_t)nstage) - 1) & 1u);
                        if (!mbar_wait_bounded(&st.empty[stage], ph, kWaitLimitNs)) *vdead = 1u;
                    }
                    if (*vdead) break;
                    const uint64_t off = (uint64_t)c * chunk_bytes;
                    const uint32_t bytes = (uint32_t)min((uint64_t)chunk_bytes, (uint64_t)geo.n16 * 16 - off);
                    fence_proxy_async();
                    mbar_arrive_expect_tx(&st.full[stage], bytes);
                    bulk_g2s(ring + (size_t)stage * chunk_bytes, reinterpret_cast<const unsigned char*>(geo.a0) + off,
                             bytes, &st.full[stage]);
                }
            }
            st.issued_lo = (uint32_t)g;
            __threadfence_block();
            *(volatile uint32_t*)&st.producer_done = 1u;
        }
        return;
    }

    // ================= consumer warps =================
    uint64_t g = 0;  // chunks consumed, in the producer's order
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
        load_params(row + stride, nT, nP, nMP, nK, nSeed);  // prefetched one row ahead
        const RowGeom geo = row_geom<ES>(a, row, chunk_bytes);
        const bool params_ok = isfinite(T) && isfinite(P) && isfinite(MP);
        const bool sampling = params_ok && T > 0.f;
        const float minp = (MP > 0.f) ? fminf(MP, 1.f) : 0.f;
        const bool listing = sampling && minp > 0.f;
        const float lt_hi = listing ? make_ctx(0.f, T, minp).L_hi * T * (1.f + 1e-5f) : 0.f;

        // ragged head/tail: loads issued now, used after the last chunk
        const int nx = geo.nhead + geo.ntail;
        float xv = -INFINITY;
        int32_t xidx = 0;
        if (tid < nx) {
            xidx = (tid < geo.nhead) ? tid : (int32_t)(a.V - geo.ntail + (tid - geo.nhead));
            xv = E::load1(geo.rowp, xidx);
        }

        auto list_token = [&](float z, int32_t i) {
            const uint32_t slot = atomicAdd(&st.lcount, 1u);
            if (slot < (uint32_t)kStreamList) {
                st.lkey[slot] = fkey(z);
                st.lidx[slot] = (uint32_t)i;
            }
        };
        auto nolist = [](float, int32_t) {};
        auto thr_of = [&](float m) -> float {
            if (!(listing && m > -INFINITY && m < INFINITY)) return INFINITY;
            const float t = list_threshold(m, lt_hi);
            return isnan(t) ? INFINITY : t;
        };

        float wrun = -INFINITY;  // this warp's running maximum over the row (same in all its lanes)
        bool dead = *vdead != 0;
        for (int c = 0; c < geo.nchunks; ++c, ++g) {
            const int stage = (int)(g % (uint64_t)nstage);
            const uint32_t parity = (uint32_t)((g / (uint64_t)nstage) & 1u);
            const uint64_t off = (uint64_t)c * chunk_bytes;
            const int nv = (int)min((uint64_t)(chunk_bytes / 16), (uint64_t)geo.n16 - off / 16);
            const uint4* cv = reinterpret_cast<const uint4*>(ring + (size_t)stage * chunk_bytes);
            const int32_t e0 = geo.nhead + (int32_t)(off / ES);
            if (!dead && !mbar_wait_bounded(&st.full[stage], parity, kWaitLimitNs)) {
                dead = true;
                *vdead = 1u;
            }
            dead = __any_sync(0xFFFFFFFFu, dead);
            if (!dead) {
                float cm;
                if (c == 0) {
                    // first chunk: this warp's own maximum over its part sets its first threshold
                    wrun = warp_max_nan(scan_max_list<TIn, false>(cv, nv, e0, INFINITY, nolist));
                    const float mref = fmax_nan(wrun, key_to_float(*(volatile uint32_t*)&st.runkey));
                    if (listing) (void)scan_max_list<TIn, false>(cv, nv, e0, thr_of(mref), list_token);
                    cm = wrun;
                } else {
                    const float mref = fmax_nan(wrun, key_to_float(*(volatile uint32_t*)&st.runkey));
                    cm = warp_max_nan(scan_max_list<TIn, false>(cv, nv, e0, thr_of(mref), list_token));
                }
                wrun = fmax_nan(wrun, cm);
                if (lane == 0 && !isnan(wrun)) atomicMax(&st.runkey, fkey(wrun));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.empty[stage]);
        }

        // ---- the ragged elements, then the row's exact maximum
        float xm = (tid < nx) ? xv : -INFINITY;
        xm = fmax_nan(wrun, warp_max_nan(xm));
        if (lane == 0) st.wmax[warp] = xm;
        if (tid < nx) {
            s.xz[tid] = xv;
            s.xi[tid] = xidx;
        }
        if (tid == 0) s.nx = nx;
        const bool cta_dead = cta_sync_or(dead || *vdead) != 0;
        float zmax = st.wmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) zmax = fmax_nan(zmax, st.wmax[w]);
        // the ragged elements are listed against the exact maximum (a threshold at least as low as
        // any running one would give, so the list stays a superset of the survivors)
        if (tid < nx && listing && xv > thr_of(zmax)) list_token(xv, xidx);

        int32_t status = kRowOk;
        if (cta_dead) status = kRowTimeout;
        else if (isnan(zmax) || zmax == INFINITY) status = kRowNan;
        else if (!params_ok) status = kRowBadParam;
        else if (zmax == -INFINITY) status = kRowAllMasked;

        float* prow = a.out_probs ? a.out_probs + row * a.V : nullptr;
        GlobalRow<TIn> src;
        src.vec = reinterpret_cast<const uint4*>(geo.a0);
        src.nvec = (int)geo.n16;
        src.elem0 = geo.nhead;

        cta_sync();  // the list and the ragged elements are complete
        const uint32_t nlisted = st.lcount;
        RowResult res;
        res.token = -1;
        if (status != kRowOk) {
            if (prow)
                for (int64_t i = tid; i < a.V; i += kThreads) prow[i] = 0.f;
            if (tid == 0) write_row(a, row, -1, status, __uint_as_float(0x7FC00000u), 0);
        } else if (T <= 0.f) {
            // greedy: lowest index of the maximum ("Implement batched top-p sampling with
            // temperature", 'A strong answer': temperature 0 means greedy, ties to the lowest index)
            uint32_t mi = 0xFFFFFFFFu;
            src.for_each(s, [&](float z, int32_t i) {
                if (z == zmax) mi = min(mi, (uint32_t)i);
            });
            mi = block_min_u32(mi, s);
            if (prow)
                for (int64_t i = tid; i < a.V; i += kThreads) prow[i] = ((uint32_t)i == mi) ? 1.f : 0.f;
            if (tid == 0) write_row(a, row, (int32_t)mi, kRowOk, zmax, 1);
        } else {
            const RowCtx r = make_ctx(zmax, T, minp);
            const float zc = minp_threshold(r);
            const bool topk_on = (K > 0) && ((int64_t)K < a.V);
            RaceCtx rc;
            rc.k0 = (uint32_t)seed;
            rc.k1 = (uint32_t)(seed >> 32);
            rc.row = (uint32_t)row;
            rc.s_lo = (uint32_t)a.step;
            rc.s_hi = (uint32_t)(a.step >> 32);
            // every survivor is on the list: filter it exactly against the true maximum
            bool fast = listing && nlisted <= (uint32_t)kStreamList;
            if (fast) {
                if (tid == 0) s.ncand = 0;
                cta_sync();
                for (uint32_t t = tid; t < nlisted; t += kThreads) {
                    const uint32_t key = st.lkey[t];
                    const float z = key_to_float(key);
                    if (z > zc && minp_ok(r, z, dist(r, z))) {
                        const uint32_t slot = atomicAdd(&s.ncand, 1u);
                        if (slot < (uint32_t)kCand) s.u.cd.sbuf[slot] = sb_make(key, st.lidx[t]);
                    }
                }
                cta_sync();
                fast = s.ncand <= (uint32_t)kCand;
            }
            if (fast) {
                res = resolve_candidates(s, r, rc, s.ncand, topk_on, K, P);
                if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
            } else {
                SoloTopo topo;
                res = general_path(topo, s, src, r, zc, topk_on, K, P, rc, prow);
            }
            if (tid == 0) write_row(a, row, res.token, kRowOk, key_to_float(res.key_cut), (int32_t)res.nk);
        }
        cta_sync();  // everyone is done with the row's shared state
        if (tid == 0) {
            st.lcount = 0;
            st.runkey = key_neg_inf;
        }
        cta_sync();
    }

    // After a timeout, copies still in flight must land before the shared memory is released.
    if (tid == 0 && *vdead) {
        const uint64_t t0 = globaltimer_ns();
        while (!*(volatile uint32_t*)&st.producer_done && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
        // the last phase issued on each stage completes only once every copy into it has landed
        const uint64_t issued = st.issued_lo;
        const uint64_t q0 = issued > (uint64_t)nstage ? issued - (uint64_t)nstage : 0;
        for (uint64_t q = q0; q < issued; ++q)
            (void)mbar_wait_bounded(&st.full[q % (uint64_t)nstage], (uint32_t)((q / (uint64_t)nstage) & 1u),
                                    kWaitLimitNs);
    }
}

}  // namespace tps
