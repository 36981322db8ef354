// tps_cluster.cuh -- the cluster sampler: a thread-block cluster per row, the row held in the
// cluster's shared memory.  Used when the batch is too small to fill the GPU with whole rows, and
// for the rows without min-p of a large batch (next to the streaming kernel), whose general path
// makes several passes over the row: on-chip here.
//
// Each of the C CTAs bulk-copies one contiguous 16-byte-aligned slice of the row from HBM into its
// own shared memory (one read of the row, no multicast); the ragged head and tail of an unaligned
// row are fetched with plain loads.  Each CTA takes its local maximum and lists the tokens that
// min-p, measured against that local maximum, does not already reject -- a superset of the row's
// survivors, because the global maximum is at least the local one.  One exchange through
// distributed shared memory gives the global maximum and the lists; every CTA then filters the
// lists exactly and resolves the row (top-k, top-p, race).  Rows whose lists overflow, or rows
// without min-p, take the general path over the slices.
#pragma once

#include "tps_common.cuh"

namespace tps {

// Per-CTA inbox of the cluster exchange: slot q holds CTA q's maximum, timeout flag, list size
// (0xFFFFFFFF: no complete list) and, for lists of at most kInbox tokens, the listed tokens.
constexpr int kInbox = 64;
constexpr int kMaxClusterCTAs = 16;
struct Inbox {
    float max[kMaxClusterCTAs];
    uint32_t timeout[kMaxClusterCTAs];
    uint32_t cnt[kMaxClusterCTAs];
    uint32_t key[kMaxClusterCTAs][kInbox];
    uint32_t idx[kMaxClusterCTAs][kInbox];
};

// ---------------------------------------------------------------------------------------------
// One row sampled by the cluster (every thread of every CTA of the cluster calls it with the same
// row).  Returns false when a bounded wait gave up: the row is reported TIMEOUT and the caller must
// not reuse the shared memory for another row.
// ---------------------------------------------------------------------------------------------
template <typename TIn>
__device__ __forceinline__ bool cluster_row(const Args& a, ClusterTopo& topo, Shared& s, Inbox* inbox,
                                            unsigned char* dsmem, int64_t row)
{
    using E = Elem<TIn>;
    constexpr int EPV = E::kPerVec;
    constexpr int ES = E::kBytes;
    cg::cluster_group& cluster = topo.g;
    const uint32_t C = topo.C;
    const uint32_t rank = topo.rank;
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;

    // ---- geometry: the aligned interior of the row in 16-byte vectors, split evenly over the CTAs
    const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + row * a.ld * ES;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(rowp), g1 = g0 + (uintptr_t)a.V * ES;
    uintptr_t a0 = (g0 + 15) & ~(uintptr_t)15, a1 = g1 & ~(uintptr_t)15;
    int64_t nhead, ntail;
    if (a1 <= a0) {
        a0 = a1 = g1;
        nhead = a.V;
        ntail = 0;
    } else {
        nhead = (int64_t)(a0 - g0) / ES;
        ntail = (int64_t)(g1 - a1) / ES;
    }
    const int64_t n16 = (int64_t)(a1 - a0) / 16;
    const int64_t v_lo = n16 * rank / C, v_hi = n16 * (rank + 1) / C;
    const int nvec = (int)(v_hi - v_lo);
    const uint32_t bytes = (uint32_t)nvec * 16u;
    Slice<TIn> sl;
    sl.vec = reinterpret_cast<const uint4*>(dsmem);
    sl.nvec = nvec;
    sl.elem0 = nhead + v_lo * EPV;

    // ---- stage the slice: one bulk copy (in 32 KB pieces) completing on an mbarrier
    const int my_head = (rank == 0) ? (int)nhead : 0;
    const int my_tail = (rank == C - 1) ? (int)ntail : 0;
    if (tid == 0) {
        s.nx = my_head + my_tail;
        if (bytes > 0) {
            fence_proxy_async();  // the previous row's reads of this slice come first
            mbar_init(&s.mbar, 1);
            mbar_arrive_expect_tx(&s.mbar, bytes);
            const unsigned char* src = reinterpret_cast<const unsigned char*>(a0) + v_lo * 16;
            for (uint32_t off = 0; off < bytes; off += 32768u)
                bulk_g2s(dsmem + off, src + off, min(32768u, bytes - off), &s.mbar);
        }
    }
    if (tid < my_head) {
        s.xz[tid] = E::load1(rowp, tid);
        s.xi[tid] = tid;
    } else if (tid < my_head + my_tail) {
        const int64_t i = a.V - ntail + (tid - my_head);
        s.xz[tid] = E::load1(rowp, i);
        s.xi[tid] = (int32_t)i;
    }
    // per-row parameters (read while the copy is in flight)
    const float T = a.temperature[row];
    const float P = a.top_p[row];
    const float MP = a.min_p[row];
    const int32_t K = a.top_k[row];
    const uint64_t seed = a.seed[row];
    const bool params_ok = isfinite(T) && isfinite(P) && isfinite(MP);
    const bool sampling = params_ok && T > 0.f;
    const float minp = (MP > 0.f) ? fminf(MP, 1.f) : 0.f;
    cta_sync();  // mbarrier initialised, extras stored
    uint32_t timed_out = 0;
    if (bytes > 0 && !mbar_wait_bounded(&s.mbar, 0, kWaitLimitNs)) timed_out = 1;
    timed_out = cta_sync_or(timed_out) ? 1u : 0u;

    // ---- A: local maximum with NaN propagation (a NaN anywhere makes the maximum NaN)
    auto nolist = [](float, int32_t) {};
    float vmax = -INFINITY;
    if (!timed_out) {
        vmax = scan_max_list<TIn, false>(sl.vec, sl.nvec, (int32_t)sl.elem0, INFINITY, nolist);
        for (int x = tid; x < s.nx; x += kThreads) vmax = fmax_nan(vmax, s.xz[x]);
    }
    vmax = warp_max_nan(vmax);
    if (lane == 0) s.rf[tid >> 5] = vmax;
    cta_sync();
    float mloc = s.rf[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) mloc = fmax_nan(mloc, s.rf[w]);

    // ---- B (local): list every token above a threshold that min-p relative to the LOCAL maximum
    //      already rejects; the global maximum is >= the local one, so the lists cover every
    //      survivor of the row.  Without min-p nothing can be excluded and no list is built.
    const bool local_ok = sampling && !timed_out && minp > 0.f && mloc > -INFINITY && mloc < INFINITY;
    uint32_t nlisted = 0xFFFFFFFFu;  // "no complete list"
    if (sampling && !timed_out && minp > 0.f && mloc == -INFINITY) nlisted = 0;  // nothing finite here
    if (local_ok) {
        const float zc_loc = list_threshold(mloc, make_ctx(0.f, T, minp).L_hi * T * (1.f + 1e-5f));
        if (tid == 0) s.ncand = 0;
        cta_sync();
        if (zc_loc > -INFINITY) {
            auto list_token = [&](float z, int32_t i) {
                const uint32_t slot = atomicAdd(&s.ncand, 1u);
                if (slot < (uint32_t)kCand) {
                    s.ckey[slot] = fkey(z);
                    s.cidx[slot] = (uint32_t)i;
                }
            };
            (void)scan_max_list<TIn, false>(sl.vec, sl.nvec, (int32_t)sl.elem0, zc_loc, list_token);
            for (int x = tid; x < s.nx; x += kThreads)
                if (s.xz[x] > zc_loc) list_token(s.xz[x], s.xi[x]);
            cta_sync();
            nlisted = s.ncand;
        }
    }
    if (tid == 0) s.pub_gcnt = min(nlisted, (uint32_t)kCand);
    // Push this CTA's maximum, timeout flag, list size and (a list of at most kInbox tokens) the
    // listed tokens into slot `rank` of every CTA's inbox: after the barrier each CTA has the whole
    // exchange in its own shared memory (longer lists are read remotely after the barrier).
    {
        const uint32_t np = (nlisted <= (uint32_t)kInbox) ? nlisted : 0u;
        const uint32_t per = np + 1u, items = C * per;
        for (uint32_t it = (uint32_t)tid; it < items; it += kThreads) {
            const uint32_t d = it / per, i = it - d * per;
            Inbox* ib = cluster.map_shared_rank(inbox, d);
            if (i == np) {
                ib->max[rank] = mloc;
                ib->timeout[rank] = timed_out;
                ib->cnt[rank] = nlisted;
            } else {
                ib->key[rank][i] = s.ckey[i];
                ib->idx[rank][i] = s.cidx[i];
            }
        }
    }
    cluster.sync();
    if (tid < 32) {
        float m = -INFINITY;
        uint32_t to = 0, nl = 0, cnt = 0, bad = 0;
        if (lane < C) {
            m = inbox->max[lane];
            to = inbox->timeout[lane];
            nl = inbox->cnt[lane];
            bad = nl > (uint32_t)kCand;
            cnt = bad ? 0u : nl;
        }
        uint32_t inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if ((int)lane >= o) inc += y;
        }
        if (lane < C) {
            s.goff[lane] = inc - cnt;
            s.gcnt[lane] = cnt;
        }
        m = warp_max_nan(m);
        to = warp_max_u32(to);
        bad = warp_max_u32(bad);
        if (lane == 31) s.gtotal = inc;
        if (lane == 0) {
            s.bf[0] = m;
            s.bu[0] = to;
            s.bu[1] = bad;
        }
    }
    cta_sync();
    const float zmax = s.bf[0];
    const uint32_t cl_timeout = s.bu[0];
    const bool lists_complete = s.bu[1] == 0;  // every CTA listed all its candidates

    int32_t status = kRowOk;
    if (cl_timeout) status = kRowTimeout;
    else if (isnan(zmax) || zmax == INFINITY) status = kRowNan;
    else if (!params_ok) status = kRowBadParam;
    else if (zmax == -INFINITY) status = kRowAllMasked;

    float* prow = a.out_probs ? a.out_probs + row * a.V : nullptr;
    const bool writer = (rank == 0) && (tid == 0);

    if (status != kRowOk) {
        if (prow) {
            for (int64_t i = sl.elem0 + tid; i < sl.elem0 + (int64_t)nvec * EPV; i += kThreads) prow[i] = 0.f;
            for (int x = tid; x < s.nx; x += kThreads) prow[s.xi[x]] = 0.f;
        }
        if (writer) write_row(a, row, -1, status, __uint_as_float(0x7FC00000u), 0);
        if (rank == 0) write_top_single(a, row, -1, tid, kThreads);
        // A copy still in flight after a timeout must land before the shared memory is released.
        if (timed_out && bytes > 0) (void)mbar_wait_bounded(&s.mbar, 0, kWaitLimitNs);
        cluster.sync();
        return !cl_timeout;
    }

    // ---- greedy branch: lowest index of the maximum ("Implement batched top-p sampling with
    //      temperature", 'A strong answer': temperature 0 means greedy, ties to the lowest index)
    if (T <= 0.f) {
        uint32_t mi = 0xFFFFFFFFu;
        sl.for_each(s, [&](float z, int32_t i) {
            if (z == zmax) mi = min(mi, (uint32_t)i);
        });
        mi = block_min_u32(mi, s);
        if (tid == 0) s.pub_minidx = mi;
        cluster.sync();
        if (tid < 32) {
            uint32_t m = (lane < C) ? *cluster.map_shared_rank(&s.pub_minidx, lane) : 0xFFFFFFFFu;
            m = warp_min_u32(m);
            if (lane == 0) s.bu[2] = m;
        }
        cta_sync();
        const uint32_t arg = s.bu[2];
        if (prow) sl.for_each(s, [&](float, int32_t i) { prow[i] = ((uint32_t)i == arg) ? 1.f : 0.f; });
        if (writer) write_row(a, row, (int32_t)arg, kRowOk, zmax, 1, 0.f);  // one-hot: ln P = 0
        if (rank == 0) write_top_single(a, row, (int32_t)arg, tid, kThreads);
        cluster.sync();
        return true;
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


    if (lists_complete) {
        // ================= fast path: every survivor is on some CTA's list =================
        // Gather the lists, keeping the survivors of min-p against the global maximum (the lists
        // were cut against each CTA's own maximum, so they may be longer).  Every CTA gathers the
        // same union, so all take the same branch below.
        if (tid == 0) s.ncand = 0;
        cta_sync();
        const uint32_t total = s.gtotal;
        for (uint32_t e = (uint32_t)tid; e < total; e += kThreads) {
            uint32_t rr = 0;
            while (rr + 1 < C && s.goff[rr + 1] <= e) ++rr;
            const uint32_t off = e - s.goff[rr];
            const bool local = inbox->cnt[rr] <= (uint32_t)kInbox;  // pushed before the barrier
            const uint32_t key = local ? inbox->key[rr][off] : *cluster.map_shared_rank(&s.ckey[off], rr);
            const uint32_t idx = local ? inbox->idx[rr][off] : *cluster.map_shared_rank(&s.cidx[off], rr);
            const float z = key_to_float(key);
            if (z > zc && minp_ok(r, z, dist(r, z))) {
                const uint32_t slot = atomicAdd(&s.ncand, 1u);
                if (slot < (uint32_t)kCand) s.u.cd.sbuf[slot] = sb_make(key, idx);
            }
        }
        cta_sync();
    }
    if (lists_complete && s.ncand <= (uint32_t)kCand) {
        cluster_arrive();  // no more remote reads by this CTA; waited for just before exit
        const uint32_t n = s.ncand;
        const RowResult res = resolve_candidates(s, r, rc, n, topk_on, K, P);
        const uint32_t key_cut = res.key_cut;
        const uint64_t NK = res.nk, ZK = res.zk;
        const int32_t token = res.token;
        if (prow) write_probs(sl, s, r, key_cut, ZK, prow);
        if (writer) write_row(a, row, token, kRowOk, key_to_float(key_cut), (int32_t)NK, token_logprob<TIn>(a, r, row, token, ZK));
        if (rank == 0) write_top(a, r, row, s.u.cd.sbuf, NK, ZK, tid, kThreads);  // sbuf is sorted
        cluster_wait();  // every CTA has finished reading this CTA's lists
        return true;
    }

    // ================= general path: survivors against the global maximum =================
    // (also when more than kCand listed tokens survive; its first barrier is a cluster barrier)
    const RowResult res = general_path(topo, s, sl, r, zc, topk_on, K, P, rc, prow, wants_zk(a));
    if (writer)
        write_row(a, row, res.token, kRowOk, key_to_float(res.key_cut), (int32_t)res.nk,
                  token_logprob<TIn>(a, r, row, res.token, res.zk));
    general_top(topo, s, sl, r, zc, res.nk, res.zk, a, row, rank == 0);
    topo.sync();  // keep this CTA's shared memory alive until every remote read is done
    return true;
}

// A failed row's outputs (token -1, cutoff NaN, kept 0, zero probabilities); all CTA threads call it.
__device__ __forceinline__ void fail_row(const Args& a, int64_t row, int32_t status)
{
    if (a.out_probs)
        for (int64_t i = threadIdx.x; i < a.V; i += kThreads) a.out_probs[row * a.V + i] = 0.f;
    if (threadIdx.x == 0) write_row(a, row, -1, status, __uint_as_float(0x7FC00000u), 0);
    write_top_single(a, row, -1, threadIdx.x, kThreads);
}

// ---------------------------------------------------------------------------------------------
// The kernel.  Grid: clusters of C CTAs along x.  With a.route == kRouteAll cluster q samples row q
// (one cluster per row).  With kRouteList the kernel runs behind the streaming kernel of a split
// batch (as its programmatic dependent): it waits for that kernel to finish, then its clusters
// claim the rows it listed in the scratch one at a time, so rows of very different cost spread
// over the clusters by themselves.
// ---------------------------------------------------------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kThreads, 2) sample_rows_kernel(const Args a)
{
    extern __shared__ __align__(128) unsigned char dsmem[];
    ClusterTopo topo;
    Shared& s = *reinterpret_cast<Shared*>(dsmem + a.slice_cap);
    topo.hr = reinterpret_cast<uint32_t*>(dsmem + a.slice_cap + sizeof(Shared));  // cluster-wide fine counts
    int32_t* rows = reinterpret_cast<int32_t*>(dsmem + a.slice_cap + sizeof(Shared) + 2 * kFineBins * sizeof(uint32_t));
    Inbox* inbox = reinterpret_cast<Inbox*>(reinterpret_cast<unsigned char*>(rows) + kThreads * sizeof(int32_t));
    const int64_t cid = (int64_t)(blockIdx.x / topo.C);
    const int tid = threadIdx.x;
    if (a.route != kRouteList) {
        if (cid < a.B) (void)cluster_row<TIn>(a, topo, s, inbox, dsmem, cid);
        return;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the streaming kernel has listed every row
    const ScratchView sv(a);
    const uint32_t nlisted = __ldcg(&sv.hdr->ngen);
    bool alive = true;
    for (;;) {
        if (topo.rank == 0 && tid == 0) s.pub_claim = atomicAdd(&sv.hdr->gclaim, 1u);
        topo.sync();
        const uint32_t k = *topo.map(&s.pub_claim, 0u);
        topo.sync();  // every CTA has read the claim before rank 0 takes the next one
        if (k >= nlisted) break;
        const int64_t row = __ldcg(&sv.genlist[k]);
        if (alive) alive = cluster_row<TIn>(a, topo, s, inbox, dsmem, row);
        else if (topo.rank == 0) fail_row(a, row, kRowTimeout);
    }
}

}  // namespace tps
