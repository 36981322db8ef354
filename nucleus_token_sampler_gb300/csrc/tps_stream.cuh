// tps_stream.cuh -- the streaming sampler: one persistent CTA per SM, whole rows streamed through a
// ring of bulk-copied chunks.  Used when the batch has enough rows to fill the GPU.
//
// Three kinds of warps, so that neither the HBM stream nor the scan ever waits for a row's
// resolution:
//   * one producer warp keeps a 3 x 64 KB ring full: as soon as a stage is released it bulk-copies
//     the next chunk of the CTA's next row into it (`cp.async.bulk` into this CTA's shared memory,
//     completed on the stage's "full" mbarrier);
//   * eight scanner warps read the chunks and release each stage through its "empty" mbarrier.
//     While a row streams, each warp keeps its running maximum (pooled across warps through an
//     atomic maximum) and lists every token that min-p, measured against that running maximum,
//     does not already reject -- a superset of the row's survivors, since the maximum only grows.
//     At the end of the row they hand the list and their maxima over in one of two row slots and
//     go straight on to the next row;
//   * one resolver warp takes each finished slot: the exact maximum, the exact min-p filter of the
//     list, the top-k and top-p cuts and the race, then frees the slot.
// Rows the resolver cannot finish alone (no min-p, an overflowing list, more than 256 survivors,
// or a probability row to write) are queued back to the scanners, which take them between rows
// with the block-wide general path over the row in global memory (just streamed, so mostly L2).
#pragma once

#include "tps_common.cuh"

namespace tps {

constexpr int kMaxStages = 8;
constexpr int kStreamThreads = kThreads + 64;  // scanner warps + resolver warp + producer warp
constexpr int kResolverWarp = kWarps;
constexpr int kProducerWarp = kWarps + 1;
constexpr int kSlotList = 1024;                // candidate list of one row slot
constexpr int kTaskQueue = 16;                 // rows handed back to the scanners

// One row handed from the scanners to the resolver.
struct RowSlot {
    uint32_t lcount;             // tokens listed (may exceed kSlotList)
    uint32_t runkey;             // order-preserving key of the pooled running maximum
    float wmax[kWarps];          // per-scanner-warp maxima (NaN-propagating)
    uint32_t lkey[kSlotList];    // listed tokens: logit key and index
    uint32_t lidx[kSlotList];
};

// Work the resolver hands back to the scanners.
enum TaskKind : uint32_t { kTaskGeneral = 1, kTaskGreedy = 2, kTaskProbs = 3, kTaskZero = 4 };
struct Task {
    uint32_t kind;
    uint32_t key_cut;
    int64_t row;
    uint64_t zk;
    float zmax;
};

struct StreamState {
    uint64_t full[kMaxStages];   // stage holds its chunk (arrive + transaction bytes)
    uint64_t empty[kMaxStages];  // every scanner warp is done with the stage
    uint64_t slot_full[2];       // every scanner warp has handed the slot over
    uint64_t slot_free[2];       // the resolver is done with the slot
    uint32_t dead;               // a bounded wait gave up: streaming stops
    uint32_t producer_done;      // the producer has left its loop
    uint32_t issued_lo;          // chunks issued (low 32 bits), valid once producer_done is set
    uint32_t resolver_done;      // the resolver has finished every row of this CTA
    uint32_t q_head, q_tail;     // task queue (the resolver pushes, the scanners pop)
    uint32_t q_seen;             // scanners: a value broadcast by thread 0
    Task q[kTaskQueue];
    // resolver scratch (one warp): survivors, sorted survivors, mass prefixes
    alignas(16) uint64_t rbuf[kCand];
    uint64_t rsorted[kCand];
    uint64_t rpre[kCand + 1];
    RowSlot slot[2];
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

// The largest float below m (m finite).
__device__ __forceinline__ float next_down(float m)
{
    if (m == 0.f) return -__uint_as_float(1u);
    const uint32_t b = __float_as_uint(m);
    return __uint_as_float(m > 0.f ? b - 1u : b + 1u);
}

struct RowParams {
    float T, P, MP;
    int32_t K;
    uint64_t seed;
};

__device__ __forceinline__ RowParams load_params(const Args& a, int64_t row)
{
    RowParams p;
    p.T = a.temperature[row];
    p.P = a.top_p[row];
    p.MP = a.min_p[row];
    p.K = a.top_k[row];
    p.seed = a.seed[row];
    return p;
}

__device__ __forceinline__ bool params_ok(const RowParams& p)
{
    return isfinite(p.T) && isfinite(p.P) && isfinite(p.MP);
}

__device__ __forceinline__ float clamp_minp(float MP) { return (MP > 0.f) ? fminf(MP, 1.f) : 0.f; }

__device__ __forceinline__ RaceCtx race_ctx(const Args& a, int64_t row, uint64_t seed)
{
    RaceCtx rc;
    rc.k0 = (uint32_t)seed;
    rc.k1 = (uint32_t)(seed >> 32);
    rc.row = (uint32_t)row;
    rc.s_lo = (uint32_t)a.step;
    rc.s_hi = (uint32_t)(a.step >> 32);
    return rc;
}

// Whether this kernel leaves the row to the cluster kernel (a split batch).
__device__ __forceinline__ bool skip_row(const Args& a, int64_t row)
{
    return a.route == kRouteStream && routed_to_cluster(a.temperature[row], a.top_p[row], a.min_p[row]);
}

// The scanners' block-wide handling of one queued row (all kThreads scanner threads call it).
template <typename TIn>
__device__ void run_task(const Args& a, Shared& s, const Task& t, uint32_t chunk_bytes)
{
    constexpr int ES = Elem<TIn>::kBytes;
    const int tid = threadIdx.x;
    const int64_t row = t.row;
    const RowGeom geo = row_geom<ES>(a, row, chunk_bytes);
    const int nx = geo.nhead + geo.ntail;
    cta_sync();  // the previous user of s.xz / s.nx is done
    if (tid < nx) {
        const int32_t xi = (tid < geo.nhead) ? tid : (int32_t)(a.V - geo.ntail + (tid - geo.nhead));
        s.xz[tid] = Elem<TIn>::load1(geo.rowp, xi);
        s.xi[tid] = xi;
    }
    if (tid == 0) s.nx = nx;
    cta_sync();
    GlobalRow<TIn> src;
    src.vec = reinterpret_cast<const uint4*>(geo.a0);
    src.nvec = (int)geo.n16;
    src.elem0 = geo.nhead;
    float* prow = a.out_probs ? a.out_probs + row * a.V : nullptr;
    const RowParams p = load_params(a, row);
    if (t.kind == kTaskZero) {
        for (int64_t i = tid; i < a.V; i += kThreads) prow[i] = 0.f;
        return;
    }
    if (t.kind == kTaskGreedy) {
        // greedy: lowest index of the maximum ("Implement batched top-p sampling with temperature",
        // 'A strong answer': temperature 0 means greedy, ties to the lowest index)
        uint32_t mi = 0xFFFFFFFFu;
        const float zmax = t.zmax;
        src.for_each(s, [&](float z, int32_t i) {
            if (z == zmax) mi = min(mi, (uint32_t)i);
        });
        mi = block_min_u32(mi, s);
        if (prow)
            for (int64_t i = tid; i < a.V; i += kThreads) prow[i] = ((uint32_t)i == mi) ? 1.f : 0.f;
        if (tid == 0) write_row(a, row, (int32_t)mi, kRowOk, zmax, 1, 0.f);
        write_top_single(a, row, (int32_t)mi, tid, kThreads);
        return;
    }
    const float minp = clamp_minp(p.MP);
    const RowCtx r = make_ctx(t.zmax, p.T, minp);
    if (t.kind == kTaskProbs) {
        write_probs(src, s, r, t.key_cut, t.zk, prow);
        return;
    }
    // kTaskGeneral
    const float zc = minp_threshold(r);
    const bool topk_on = (p.K > 0) && ((int64_t)p.K < a.V);
    SoloTopo topo;
    const RowResult res =
        general_path(topo, s, src, r, zc, topk_on, p.K, p.P, race_ctx(a, row, p.seed), prow, wants_zk(a));
    if (tid == 0)
        write_row(a, row, res.token, kRowOk, key_to_float(res.key_cut), (int32_t)res.nk,
                  token_logprob<TIn>(a, r, row, res.token, res.zk));
    general_top(topo, s, src, r, zc, res.nk, res.zk, a, row, true);
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&st.slot_full[i], kWarps);
            mbar_init(&st.slot_free[i], 1);
            st.slot[i].lcount = 0;
            st.slot[i].runkey = key_neg_inf;
        }
        st.dead = 0;
        st.producer_done = 0;
        st.issued_lo = 0;
        st.resolver_done = 0;
        st.q_head = st.q_tail = 0;
    }
    __syncthreads();  // the only CTA-wide barrier

    // ================= producer warp =================
    if (warp == kProducerWarp) {
        if (lane == 0) {
            uint64_t g = 0;
            bool skip_next = skip_row(a, first);
            for (int64_t row = first; row < B && !*vdead; row += stride) {
                const bool skip = skip_next;
                if (row + stride < B) skip_next = skip_row(a, row + stride);
                if (skip) continue;
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

    // ================= resolver warp =================
    if (warp == kResolverWarp) {
        auto push = [&](const Task& t) {  // lane 0 only; waits (bounded) for queue space
            const uint64_t t0 = globaltimer_ns();
            while (*(volatile uint32_t*)&st.q_tail - *(volatile uint32_t*)&st.q_head >= (uint32_t)kTaskQueue) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    *vdead = 1u;
                    return;
                }
                __nanosleep(200);
            }
            const uint32_t tail = *(volatile uint32_t*)&st.q_tail;
            st.q[tail % kTaskQueue] = t;
            __threadfence_block();
            *(volatile uint32_t*)&st.q_tail = tail + 1;
        };
        int64_t j = 0;  // rows of this CTA sampled so far
        for (int64_t row = first; row < B; row += stride) {
            if (skip_row(a, row)) continue;
            const int sl = (int)(j & 1);
            RowSlot& slot = st.slot[sl];
            bool ok = mbar_wait_bounded(&st.slot_full[sl], (uint32_t)((j >> 1) & 1), kWaitLimitNs);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) *vdead = 1u;
            float zmax = slot.wmax[0];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) zmax = fmax_nan(zmax, slot.wmax[w]);
            const RowParams p = load_params(a, row);
            const uint32_t nlisted = slot.lcount;
            int32_t status = kRowOk;
            if (!ok || *vdead) status = kRowTimeout;
            else if (isnan(zmax) || zmax == INFINITY) status = kRowNan;
            else if (!params_ok(p)) status = kRowBadParam;
            else if (zmax == -INFINITY) status = kRowAllMasked;
            Task t;
            t.row = row;
            t.zmax = zmax;
            t.key_cut = 0;
            t.zk = 0;
            t.kind = 0;
            if (status != kRowOk) {
                if (lane == 0) write_row(a, row, -1, status, __uint_as_float(0x7FC00000u), 0);
                write_top_single(a, row, -1, (int)lane, 32);
                if (a.out_probs) t.kind = kTaskZero;
            } else if (p.T <= 0.f) {
                // greedy: the lowest listed index holding the maximum (the list holds every token
                // that reached the running maximum), unless the list overflowed
                if (nlisted <= (uint32_t)kSlotList && !a.out_probs) {
                    uint32_t mi = 0xFFFFFFFFu;
                    for (uint32_t e = lane; e < nlisted; e += 32)
                        if (key_to_float(slot.lkey[e]) == zmax) mi = min(mi, slot.lidx[e]);
                    mi = __reduce_min_sync(0xFFFFFFFFu, mi);
                    if (lane == 0) write_row(a, row, (int32_t)mi, kRowOk, zmax, 1, 0.f);
                    write_top_single(a, row, (int32_t)mi, (int)lane, 32);
                } else {
                    t.kind = kTaskGreedy;  // a pass over the row (also writes the one-hot row)
                }
            } else {
                const float minp = clamp_minp(p.MP);
                const RowCtx r = make_ctx(zmax, p.T, minp);
                const float zc = minp_threshold(r);
                const bool topk_on = (p.K > 0) && ((int64_t)p.K < a.V);
                bool fast = minp > 0.f && nlisted <= (uint32_t)kSlotList;
                uint32_t n = 0;
                if (fast) {
                    // exact min-p filter of the list against the true maximum (ballot compaction)
                    for (uint32_t e0 = 0; e0 < nlisted; e0 += 32) {
                        const uint32_t e = e0 + lane;
                        bool keep = false;
                        uint32_t key = 0, idx = 0;
                        if (e < nlisted) {
                            key = slot.lkey[e];
                            idx = slot.lidx[e];
                            const float z = key_to_float(key);
                            keep = z > zc && minp_ok(r, z, dist(r, z));
                        }
                        const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep);
                        const uint32_t at = n + __popc(m & ((1u << lane) - 1u));
                        if (keep && at < (uint32_t)kCand) st.rbuf[at] = sb_make(key, idx);
                        n += __popc(m);
                    }
                    __syncwarp();
                    fast = n <= (uint32_t)kCand;
                }
                if (fast) {
                    const RaceCtx rc = race_ctx(a, row, p.seed);
                    const WarpResult wr = (n <= 32) ? warp_resolve(st.rbuf, r, rc, n, topk_on, p.K, p.P)
                                                    : warp_resolve_big(st.rbuf, st.rsorted, st.rpre, n, r, rc, topk_on,
                                                                       p.K, p.P);
                    if (lane == 0)
                        write_row(a, row, wr.token, kRowOk, key_to_float(wr.key_cut), (int32_t)wr.nk,
                                  token_logprob<TIn>(a, r, row, wr.token, wr.zk));
                    __syncwarp();  // the sorted survivors are visible to every lane
                    write_top(a, r, row, (n <= 32) ? st.rbuf : st.rsorted, wr.nk, wr.zk, (int)lane, 32);
                    if (a.out_probs) {
                        t.kind = kTaskProbs;
                        t.key_cut = wr.key_cut;
                        t.zk = wr.zk;
                    }
                } else {
                    t.kind = kTaskGeneral;
                }
            }
            // hand back what needs the scanners, then free the slot for row j + 2
            __syncwarp();
            if (lane == 0) {
                if (t.kind) push(t);
                slot.lcount = 0;
                slot.runkey = key_neg_inf;
                __threadfence_block();
                mbar_arrive(&st.slot_free[sl]);
            }
            __syncwarp();
            ++j;
        }
        if (lane == 0) {
            __threadfence_block();
            *(volatile uint32_t*)&st.resolver_done = 1u;
        }
        return;
    }

    // ================= scanner warps =================
    // Take every queued row (all scanner threads together) until the queue is seen empty.
    auto drain = [&]() {
        for (;;) {
            if (tid == 0) st.q_seen = *(volatile uint32_t*)&st.q_tail;
            cta_sync();
            const uint32_t tail = st.q_seen, head = st.q_head;
            cta_sync();
            if (tail == head) break;
            for (uint32_t h = head; h != tail; ++h) {
                const Task t = st.q[h % kTaskQueue];
                run_task<TIn>(a, s, t, chunk_bytes);
                cta_sync();
            }
            if (tid == 0) *(volatile uint32_t*)&st.q_head = tail;
        }
    };

    uint64_t g = 0;  // chunks consumed, in the producer's order
    RowParams nxt = load_params(a, first);
    int64_t j = 0;  // rows of this CTA sampled so far
    for (int64_t row = first; row < B; row += stride) {
        const RowParams p = nxt;
        if (row + stride < B) nxt = load_params(a, row + stride);  // prefetched one row ahead
        if (a.route == kRouteStream && routed_to_cluster(p.T, p.P, p.MP)) continue;
        drain();
        const int sl = (int)(j & 1);
        RowSlot& slot = st.slot[sl];
        bool dead = *vdead != 0;
        if (j >= 2 && !dead && !mbar_wait_bounded(&st.slot_free[sl], (uint32_t)(((j >> 1) - 1) & 1), kWaitLimitNs)) {
            dead = true;
            *vdead = 1u;
        }
        const RowGeom geo = row_geom<ES>(a, row, chunk_bytes);
        const bool ok = params_ok(p);
        const float minp = clamp_minp(p.MP);
        // listing: min-p rows list what min-p against the running maximum cannot exclude; greedy
        // rows list what reaches the running maximum (a superset of the final maximum's class)
        const bool greedy = ok && p.T <= 0.f;
        const bool listing = (ok && p.T > 0.f && minp > 0.f) || greedy;
        const float lt_hi = (listing && !greedy) ? make_ctx(0.f, p.T, minp).L_hi * p.T * (1.f + 1e-5f) : 0.f;
        auto thr_of = [&](float m) -> float {
            if (!(listing && m > -INFINITY && m < INFINITY)) return INFINITY;
            if (greedy) return next_down(m);
            const float t = list_threshold(m, lt_hi);
            return isnan(t) ? INFINITY : t;
        };
        auto list_token = [&](float z, int32_t i) {
            const uint32_t at = atomicAdd(&slot.lcount, 1u);
            if (at < (uint32_t)kSlotList) {
                slot.lkey[at] = fkey(z);
                slot.lidx[at] = (uint32_t)i;
            }
        };
        auto nolist = [](float, int32_t) {};

        // ragged head/tail (warp 0 lanes): listed unconditionally, the resolver filters them
        const int nx = geo.nhead + geo.ntail;
        float xv = -INFINITY;
        int32_t xidx = 0;
        if (tid < nx) {
            xidx = (tid < geo.nhead) ? tid : (int32_t)(a.V - geo.ntail + (tid - geo.nhead));
            xv = E::load1(geo.rowp, xidx);
        }

        float wrun = -INFINITY;  // this warp's running maximum over the row (same in all its lanes)
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
                    const float mref = fmax_nan(wrun, key_to_float(*(volatile uint32_t*)&slot.runkey));
                    if (listing) (void)scan_max_list<TIn, false>(cv, nv, e0, thr_of(mref), list_token);
                    cm = wrun;
                } else {
                    const float mref = fmax_nan(wrun, key_to_float(*(volatile uint32_t*)&slot.runkey));
                    cm = warp_max_nan(scan_max_list<TIn, false>(cv, nv, e0, thr_of(mref), list_token));
                }
                wrun = fmax_nan(wrun, cm);
                if (lane == 0 && !isnan(wrun)) atomicMax(&slot.runkey, fkey(wrun));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.empty[stage]);
        }
        // hand the row over: ragged elements (listed), this warp's maximum, arrive on the slot
        if (tid < nx) list_token(xv, xidx);
        const float xm = warp_max_nan((tid < nx) ? xv : -INFINITY);
        if (lane == 0) slot.wmax[warp] = dead ? __uint_as_float(0x7FC00000u) : fmax_nan(wrun, xm);
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            mbar_arrive(&st.slot_full[sl]);
        }
        ++j;
    }
    // keep taking queued rows until the resolver has finished every row
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        drain();
        if (tid == 0) st.q_seen = *(volatile uint32_t*)&st.resolver_done;
        cta_sync();
        const bool rdone = st.q_seen != 0;
        cta_sync();
        if (rdone) {
            drain();
            break;
        }
        if (globaltimer_ns() - t0 > 4 * kWaitLimitNs) break;  // a resolver wait has already given up
        __nanosleep(500);
    }

    // After a timeout, copies still in flight must land before the shared memory is released.
    if (tid == 0 && *vdead) {
        const uint64_t t1 = globaltimer_ns();
        while (!*(volatile uint32_t*)&st.producer_done && globaltimer_ns() - t1 < kWaitLimitNs) {
        }
        // the last phase issued on each stage completes only once every copy into it has landed
        const uint64_t issued = st.issued_lo;
        const uint64_t q0 = issued > (uint64_t)nstage ? issued - (uint64_t)nstage : 0;
        for (uint64_t q = q0; q < issued; ++q)
            (void)mbar_wait_bounded(&st.full[q % (uint64_t)nstage], (uint32_t)((q / (uint64_t)nstage) & 1u),
                                    kWaitLimitNs);
    }
    // Launched as the programmatic dependent of the cluster kernel (a split batch): this CTA -- so
    // this grid -- completes only after that kernel has, so later work in the stream sees both.
    // A no-op for an ordinary launch.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace tps
