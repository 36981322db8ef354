// tps_stream.cuh -- the streaming sampler: one persistent CTA per SM, rows streamed through a ring
// of bulk-copied chunks.  Used when the batch has enough rows to fill the GPU.
//
// Work is claimed dynamically, so SMs that stream faster take more of it and all finish within about
// one claim of each other.  A batch with several rows per SM is claimed in whole rows; a smaller one
// has every row split into segments (the host chooses, see the plan in tps_api.cu).  A CTA's first
// two claims are fixed (its block index, then that plus the grid size); later claims come from a
// counter in the call's global scratch (cleared by a small kernel launched just before this one,
// which this kernel waits for before it touches the scratch).
//
// Three kinds of warps, so that neither the HBM stream nor the scan ever waits for a row's
// resolution:
//   * one producer warp claims units of work (a whole row, or a segment of a split row) and keeps a
//     3 x 64 KB ring full: as soon as a stage is released it describes the unit's next chunk in the
//     stage and bulk-copies the chunk into it (`cp.async.bulk` into this CTA's shared memory,
//     completed on the stage's "full" mbarrier);
//   * eight scanner warps read the chunks and release each stage through its "empty" mbarrier.
//     While a unit streams, each warp keeps its running maximum (pooled across warps through an
//     atomic maximum) and lists every token that min-p, measured against that running maximum,
//     does not already reject -- a superset of the survivors, since the maximum only grows.  The
//     unit's first chunk is read twice: once for its maximum, then to list against it.  At the end
//     of the unit they hand the list and their maxima over in one of three slots and go on;
//   * two resolver warps take the finished slots, alternately.  A whole row is resolved on the spot: the exact
//     maximum, the exact min-p filter of the list, the top-k and top-p cuts and the race.  A segment
//     of a split row publishes its maximum and its exactly filtered list to the scratch and counts
//     itself on the row's counter; the resolver whose segment completes the count merges the
//     published lists against the row's maximum and resolves the row the same way.
// Rows the resolver cannot finish alone (no min-p, an overflowing list, more than 256 survivors, or
// a probability row to write) are queued back to the scanners, which take them between units with
// the block-wide general path over the row in global memory.  In a split batch (kRouteStream) rows
// without min-p are not streamed at all: the producer lists them in the scratch for the cluster
// kernel, launched behind this one.
#pragma once

#include "tps_common.cuh"

namespace tps {

constexpr int kMaxStages = 8;
constexpr int kResolvers = 2;                  // resolver warps (they take alternate units)
constexpr int kStreamThreads = kThreads + 32 * (kResolvers + 1);  // scanner warps, resolver warps, producer warp
constexpr int kResolverWarp = kWarps;          // the first resolver warp
constexpr int kProducerWarp = kWarps + kResolvers;
constexpr int kSlotList = 384;                 // candidate list of one slot
constexpr int kSlots = 3;                      // slots between the scanners and the resolvers
constexpr int kTaskQueue = 16;                 // rows handed back to the scanners
constexpr int kUnitLog = 16;                   // claims of the units most recently put in the ring
static_assert(32 * kMaxSegments <= kCand, "a merge parks 32 entries of every segment in a resolver's sort buffer");

struct RowParams {
    float T, P, MP;
    int32_t K;
    uint64_t seed;
};

// One unit of work: a whole row (nseg == 1), or segment `seg` of the nseg segments of a split row.
struct Unit {
    int64_t row;
    int32_t seg, nseg;
};

__device__ __forceinline__ int64_t total_claims(const Args& a) { return a.b_whole + a.nsplit * (int64_t)a.nseg; }

__device__ __forceinline__ Unit unit_of(const Args& a, int64_t q)
{
    Unit u;
    if (q < a.b_whole) {
        u.row = q;
        u.seg = 0;
        u.nseg = 1;
    } else {
        const int64_t k = q - a.b_whole;
        u.row = a.b_whole + k / a.nseg;
        u.seg = (int32_t)(k % a.nseg);
        u.nseg = a.nseg;
    }
    return u;
}

// What a ring stage holds, written by the producer before it starts the stage's copy (the stage's
// "full" mbarrier publishes it to the scanners with the data).
struct StageInfo {
    int64_t row;  // < 0: no more work
    int32_t seg, nseg;
    RowParams p;
};

// One unit handed from the scanners to a resolver.
struct RowSlot {
    uint32_t lcount;             // tokens listed (may exceed kSlotList)
    uint32_t runkey;             // order-preserving key of the pooled running maximum
    float wmax[kWarps];          // per-scanner-warp maxima (NaN-propagating)
    int64_t row;                 // < 0: no more work
    int32_t seg, nseg;
    RowParams p;
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

// What one resolver warp owns: its survivors, sorted survivors and mass prefixes, and the queue of
// rows it hands back to the scanners (it pushes, the scanners pop).
struct ResolverSpace {
    alignas(16) uint64_t rbuf[kCand];
    uint64_t rsorted[kCand];
    uint64_t rpre[kCand + 1];
    uint32_t q_head, q_tail;
    Task q[kTaskQueue];
};

struct StreamState {
    uint64_t full[kMaxStages];   // stage holds its chunk (arrive + transaction bytes)
    uint64_t empty[kMaxStages];  // every scanner warp is done with the stage
    uint64_t slot_full[kSlots];  // every scanner warp has handed the slot over
    uint64_t slot_free[kSlots];  // its resolver has taken what it needs from the slot
    uint32_t dead;               // a bounded wait gave up: streaming stops
    uint32_t producer_done;      // the producer has left its loop
    uint32_t issued_lo;          // chunks issued (low 32 bits), valid once producer_done is set
    uint32_t resolvers_done;     // resolver warps that have finished every unit they take
    uint32_t units_put;          // units put in the ring, valid once producer_done is set
    uint32_t withheld;           // test hook: 1 + the chunk whose copy was withheld (0: none)
    uint32_t q_seen;             // scanners: a value broadcast by thread 0
    int64_t ulog[kUnitLog];      // claims of the units put in the ring, by order of putting
    StageInfo info[kMaxStages];
    ResolverSpace rs[kResolvers];
    RowSlot slot[kSlots];
};

// Geometry of one row: aligned interior in 16-byte vectors plus a ragged head and tail.
struct RowGeom {
    const unsigned char* rowp;
    uintptr_t a0;      // 16-byte-aligned start of the interior
    int64_t n16;       // interior vectors
    int nhead, ntail;  // ragged elements before / after the interior
};

template <int ES>
__device__ __forceinline__ RowGeom row_geom(const Args& a, int64_t row)
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
    return g;
}

// A unit's share of the row's aligned interior, vectors [v_lo, v_hi), in chunks of at most
// chunk_bytes; a unit with no interior still takes one (empty) chunk, so it passes through the
// ring like any other.  Segment 0 also owns the ragged head, the last segment the ragged tail.
struct UnitGeom {
    int64_t v_lo, v_hi;
    int nchunks;
};
__device__ __forceinline__ UnitGeom unit_geom(const RowGeom& g, int seg, int nseg, uint32_t chunk_bytes)
{
    UnitGeom u;
    u.v_lo = g.n16 * seg / nseg;
    u.v_hi = g.n16 * (seg + 1) / nseg;
    const int64_t bytes = (u.v_hi - u.v_lo) * 16;
    u.nchunks = bytes > 0 ? (int)((bytes + chunk_bytes - 1) / chunk_bytes) : 1;
    return u;
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

// The scanners' block-wide handling of one queued row (all kThreads scanner threads call it).
template <typename TIn>
__device__ void run_task(const Args& a, Shared& s, const Task& t)
{
    constexpr int ES = Elem<TIn>::kBytes;
    const int tid = threadIdx.x;
    const int64_t row = t.row;
    const RowGeom geo = row_geom<ES>(a, row);
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


// A whole row's status from its maximum and parameters.
__device__ __forceinline__ int32_t row_status(float zmax, const RowParams& p)
{
    if (isnan(zmax) || zmax == INFINITY) return kRowNan;
    if (!params_ok(p)) return kRowBadParam;
    if (zmax == -INFINITY) return kRowAllMasked;
    return kRowOk;
}

// Top-k, top-p and the race over a row's survivors st.rbuf[0, n) (1 <= n <= kCand, any order), one
// warp, then the row's outputs; a probability row is left to the scanners (t).
template <typename TIn>
__device__ __forceinline__ void resolve_listed(const Args& a, ResolverSpace& st, const RowCtx& r, const RowParams& p,
                                               int64_t row, uint32_t n, Task& t)
{
    const uint32_t lane = threadIdx.x & 31;
    const bool topk_on = (p.K > 0) && ((int64_t)p.K < a.V);
    const RaceCtx rc = race_ctx(a, row, p.seed);
    const WarpResult wr = (n <= 32) ? warp_resolve(st.rbuf, r, rc, n, topk_on, p.K, p.P)
                                    : warp_resolve_big(st.rbuf, st.rsorted, st.rpre, n, r, rc, topk_on, p.K, p.P);
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
}

// What the resolver takes from a slot.  Everything it needs later is copied out of the slot -- the
// unit, the maximum, and the listed tokens that survive an exact filter, into st.rbuf -- so the slot
// is handed back to the scanners at once and the rest of the resolution (the cuts, the race, the
// partial results of a split row, the merge) never holds them up.
struct Job {
    int64_t row;
    int32_t seg, nseg;
    RowParams p;
    float zmax;      // a whole row's maximum, or a segment's own maximum
    int32_t status;  // a whole row's status (kRowOk for a segment: the merge decides)
    uint32_t n;      // survivors copied to st.rbuf (greedy: tokens equal to the maximum)
    uint32_t flags;  // PartFlag bits: the list overflowed, the row lists nothing, a wait gave up
    uint32_t mi;     // greedy: the lowest index holding the maximum among the listed tokens
};

// Take a unit from its slot (one warp).  The listed tokens are filtered exactly against m, the
// unit's maximum (a whole row's: its survivors; a segment's: a superset of the row's survivors, the
// row's maximum being at least as large), or, for a greedy row, kept when equal to m.
__device__ __forceinline__ Job take_unit(const Args& a, ResolverSpace& st, const RowSlot& slot, bool dead)
{
    const uint32_t lane = threadIdx.x & 31;
    Job jb;
    jb.row = slot.row;
    jb.seg = slot.seg;
    jb.nseg = slot.nseg;
    jb.p = slot.p;
    float m = slot.wmax[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmax_nan(m, slot.wmax[w]);
    jb.zmax = m;
    jb.n = 0;
    jb.mi = 0xFFFFFFFFu;
    const uint32_t nlisted = slot.lcount;
    const bool pok = params_ok(jb.p);
    const bool greedy = pok && jb.p.T <= 0.f;
    const float minp = clamp_minp(jb.p.MP);
    const bool listing = greedy || (pok && jb.p.T > 0.f && minp > 0.f);
    jb.flags = dead ? (uint32_t)kPartTimeout : 0u;
    if (!listing) jb.flags |= kPartUnlisted;
    if (nlisted > (uint32_t)kSlotList) jb.flags |= kPartOverflow;
    jb.status = dead ? (int32_t)kRowTimeout : (jb.nseg == 1 ? row_status(m, jb.p) : (int32_t)kRowOk);
    if (jb.flags == 0 && jb.status == kRowOk && m > -INFINITY && m < INFINITY) {
        const RowCtx r = make_ctx(m, jb.p.T, minp);
        const float zc = greedy ? m : minp_threshold(r);
        uint32_t n = 0, mi = 0xFFFFFFFFu;
        for (uint32_t e0 = 0; e0 < nlisted; e0 += 32) {
            const uint32_t e = e0 + lane;
            bool keep = false;
            uint32_t key = 0, idx = 0;
            if (e < nlisted) {
                key = slot.lkey[e];
                idx = slot.lidx[e];
                const float z = key_to_float(key);
                keep = greedy ? (z == m) : (z > zc && minp_ok(r, z, dist(r, z)));
            }
            if (keep && greedy) mi = min(mi, idx);
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, keep);
            const uint32_t at = n + __popc(b & ((1u << lane) - 1u));
            if (keep && at < (uint32_t)kCand) st.rbuf[at] = sb_make(key, idx);
            n += __popc(b);
        }
        jb.n = n;
        jb.mi = __reduce_min_sync(0xFFFFFFFFu, mi);
        if (n > (uint32_t)kCand) jb.flags |= kPartOverflow;
    }
    __syncwarp();
    return jb;
}

// Finish a whole row from its job (one warp); returns the task it leaves to the scanners.
template <typename TIn>
__device__ Task finish_row(const Args& a, ResolverSpace& st, const Job& jb)
{
    const uint32_t lane = threadIdx.x & 31;
    const int64_t row = jb.row;
    Task t;
    t.row = row;
    t.zmax = jb.zmax;
    t.key_cut = 0;
    t.zk = 0;
    t.kind = 0;
    if (jb.status != kRowOk) {
        if (lane == 0) write_row(a, row, -1, jb.status, __uint_as_float(0x7FC00000u), 0);
        write_top_single(a, row, -1, (int)lane, 32);
        if (a.out_probs) t.kind = kTaskZero;
        return t;
    }
    if (jb.p.T <= 0.f) {
        // greedy: the lowest listed index holding the maximum (the list holds every token that
        // reached the running maximum), unless the list overflowed or a one-hot row is asked for
        if (!(jb.flags & kPartOverflow) && !a.out_probs) {
            if (lane == 0) write_row(a, row, (int32_t)jb.mi, kRowOk, jb.zmax, 1, 0.f);
            write_top_single(a, row, (int32_t)jb.mi, (int)lane, 32);
        } else {
            t.kind = kTaskGreedy;  // a pass over the row (also writes the one-hot row)
        }
        return t;
    }
    if (jb.flags & (kPartOverflow | kPartUnlisted)) {
        t.kind = kTaskGeneral;
        return t;
    }
    const RowCtx r = make_ctx(jb.zmax, jb.p.T, clamp_minp(jb.p.MP));
    resolve_listed<TIn>(a, st, r, jb.p, row, jb.n, t);
    return t;
}

// Merge the published segments of a split row (one warp, run by the resolver whose segment
// completed the row's count) and resolve the row.  Partials are read through L2 (ld.global.cg): they
// were written by other SMs.
template <typename TIn>
__device__ Task merge_row(const Args& a, const ScratchView& sv, ResolverSpace& st, int64_t row, const RowParams& p)
{
    const uint32_t lane = threadIdx.x & 31;
    const int nseg = a.nseg;
    const int64_t sr = row - a.b_whole;
    // one round trip: every segment's header and its first 32 entries (parked in rsorted)
    float m = -INFINITY;
    uint32_t cnt = 0, fl = 0;
    if ((int)lane < nseg) {
        const PartHdr* h = sv.part_hdr(sr, (int)lane, nseg);
        m = __ldcg(&h->max);
        cnt = __ldcg(&h->n);
        fl = __ldcg(&h->flags);
    }
    for (int q = 0; q < nseg; ++q)
        st.rsorted[32 * q + lane] = __ldcg(reinterpret_cast<const unsigned long long*>(sv.part_ent(sr, q, nseg)) + lane);
    __syncwarp();
    const float M = warp_max_nan(m);
    const uint32_t F = __reduce_or_sync(0xFFFFFFFFu, fl);
    uint32_t inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if ((int)lane >= o) inc += y;
    }
    const uint32_t off = inc - cnt;
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, inc, 31);
    // the published entry e of the concatenation of the segments' lists
    auto entry = [&](uint32_t e) -> uint64_t {
        int s = 0;
        for (int q = 1; q < nseg; ++q)
            if (e >= __shfl_sync(0xFFFFFFFFu, off, q)) s = q;
        const uint32_t o = e - __shfl_sync(0xFFFFFFFFu, off, s);
        return o < 32u ? st.rsorted[32 * s + o]
                       : __ldcg(reinterpret_cast<const unsigned long long*>(sv.part_ent(sr, s, nseg)) + o);
    };
    Task t;
    t.row = row;
    t.zmax = M;
    t.key_cut = 0;
    t.zk = 0;
    t.kind = 0;
    const int32_t status = (F & kPartTimeout) ? (int32_t)kRowTimeout : row_status(M, p);
    if (status != kRowOk) {
        if (lane == 0) write_row(a, row, -1, status, __uint_as_float(0x7FC00000u), 0);
        write_top_single(a, row, -1, (int)lane, 32);
        if (a.out_probs) t.kind = kTaskZero;
        return t;
    }
    if (p.T <= 0.f) {
        if ((F & kPartOverflow) || a.out_probs) {
            t.kind = kTaskGreedy;
            return t;
        }
        uint32_t mi = 0xFFFFFFFFu;
        for (uint32_t e0 = 0; e0 < total; e0 += 32) {  // uniform trip count: entry() shuffles
            const uint32_t e = min(e0 + lane, total - 1);
            const uint64_t v = entry(e);
            if (e0 + lane < total && key_to_float(sb_key(v)) == M) mi = min(mi, (uint32_t)sb_idx(v));
        }
        mi = __reduce_min_sync(0xFFFFFFFFu, mi);
        if (lane == 0) write_row(a, row, (int32_t)mi, kRowOk, M, 1, 0.f);
        write_top_single(a, row, (int32_t)mi, (int)lane, 32);
        return t;
    }
    const float minp = clamp_minp(p.MP);
    if ((F & (kPartOverflow | kPartUnlisted)) || !(minp > 0.f)) {
        t.kind = kTaskGeneral;
        return t;
    }
    const RowCtx r = make_ctx(M, p.T, minp);
    const float zc = minp_threshold(r);
    uint32_t n = 0;
    for (uint32_t e0 = 0; e0 < total; e0 += 32) {
        const uint32_t e = min(e0 + lane, total - 1);
        const uint64_t v = entry(e);
        bool keep = false;
        if (e0 + lane < total) {
            const float z = key_to_float(sb_key(v));
            keep = z > zc && minp_ok(r, z, dist(r, z));
        }
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, keep);
        const uint32_t at = n + __popc(b & ((1u << lane) - 1u));
        if (keep && at < (uint32_t)kCand) st.rbuf[at] = v;
        n += __popc(b);
    }
    __syncwarp();
    if (n > (uint32_t)kCand) {
        t.kind = kTaskGeneral;
        return t;
    }
    resolve_listed<TIn>(a, st, r, p, row, n, t);
    return t;
}

// Finish a segment of a split row from its job (one warp): publish the segment's maximum and
// survivors and count the segment on the row's counter; the segment that completes the count
// merges the row.
template <typename TIn>
__device__ Task finish_segment(const Args& a, const ScratchView& sv, ResolverSpace& st, const Job& jb)
{
    const uint32_t lane = threadIdx.x & 31;
    const int64_t sr = jb.row - a.b_whole;
    PartHdr* h = sv.part_hdr(sr, jb.seg, jb.nseg);
    uint64_t* ent = sv.part_ent(sr, jb.seg, jb.nseg);
    const uint32_t n = (jb.flags & kPartOverflow) ? 0u : jb.n;
    for (uint32_t e = lane; e < n; e += 32) ent[e] = st.rbuf[e];
    if (lane == 0) {
        h->max = jb.zmax;
        h->n = n;
        h->flags = jb.flags;
    }
    __syncwarp();  // every lane's entries are written before lane 0 publishes them
    uint32_t old = 0;
    if (lane == 0) {
        __threadfence();  // (cumulative) the warp's entries are visible GPU-wide before the segment is counted
        old = atomicAdd(&sv.arrive[sr], 1u);
        __threadfence();  // and, for the last segment, the other segments' partials are visible after it
    }
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    __syncwarp();
    Task t;
    t.row = jb.row;
    t.kind = 0;
    t.key_cut = 0;
    t.zk = 0;
    t.zmax = jb.zmax;
    if (old + 1u < (uint32_t)jb.nseg) return t;
    return merge_row<TIn>(a, sv, st, jb.row, jb.p);
}

// A unit this CTA could not stream (a bounded wait gave up): its row is reported TIMEOUT -- at once
// for a whole row; for a segment, through a partial flagged kPartTimeout, so whichever CTA completes
// the row's count reports it.  One thread.
__device__ __forceinline__ void fail_unit(const Args& a, const ScratchView& sv, int64_t q)
{
    const Unit u = unit_of(a, q);
    const float qnan = __uint_as_float(0x7FC00000u);
    if (u.nseg == 1) {
        write_row(a, u.row, -1, kRowTimeout, qnan, 0);
        write_top_single(a, u.row, -1, 0, 1);
        return;
    }
    const int64_t sr = u.row - a.b_whole;
    PartHdr* h = sv.part_hdr(sr, u.seg, u.nseg);
    h->max = qnan;
    h->n = 0;
    h->flags = kPartTimeout;
    __threadfence();
    if (atomicAdd(&sv.arrive[sr], 1u) + 1u == (uint32_t)u.nseg) {
        __threadfence();
        write_row(a, u.row, -1, kRowTimeout, qnan, 0);
        write_top_single(a, u.row, -1, 0, 1);
    }
}

__device__ __forceinline__ void wait_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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
    const int64_t Q = total_claims(a);
    const ScratchView sv(a);
    const uint32_t key_neg_inf = 0x007FFFFFu;  // fkey(-inf)
    const uint64_t wait_ns = a.wait_ns;         // consumer-side wait limit (kWaitLimitNs but in tests)

    if (tid == 0) {
        // the kernel queued behind this one (the cluster kernel of a split batch) may launch now; it
        // waits for this grid to complete before it reads what this kernel writes
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&st.full[i], 1);
            mbar_init(&st.empty[i], kWarps);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&st.slot_full[i], kWarps);
            mbar_init(&st.slot_free[i], 1);
            st.slot[i].lcount = 0;
            st.slot[i].runkey = key_neg_inf;
        }
        st.dead = 0;
        st.producer_done = 0;
        st.issued_lo = 0;
        st.resolvers_done = 0;
        st.units_put = 0;
        st.withheld = 0;
        for (int i = 0; i < kResolvers; ++i) st.rs[i].q_head = st.rs[i].q_tail = 0;
    }
    __syncthreads();  // the only CTA-wide barrier

    // ================= producer warp =================
    if (warp == kProducerWarp) {
        if (lane == 0) {
            uint64_t g = 0;
            uint32_t nput = 0;
            bool waited = false;
            // The scratch is cleared by the kernel this one is launched behind: wait for it (and
            // everything before it) before the first access.  Logits and parameters may be read
            // earlier: that kernel started only after all earlier work had completed.
            // This CTA's claims: its block index, then (fixed) its block index + gridDim.x, then the
            // counter's, from 2 gridDim.x on.  Every path that takes a unit takes it from here.
            uint32_t nclaims = 1;
            auto claim_counter = [&]() -> int64_t {
                if (!waited) {
                    wait_prerequisite();
                    waited = true;
                }
                return 2 * (int64_t)gridDim.x + (int64_t)atomicAdd(&sv.hdr->claim, 1u);
            };
            auto claim = [&]() -> int64_t {
                if (nclaims++ == 1) return (int64_t)blockIdx.x + (int64_t)gridDim.x;
                return claim_counter();
            };
            auto list_for_cluster = [&](int64_t row) {
                if (!waited) {
                    wait_prerequisite();
                    waited = true;
                }
                sv.genlist[atomicAdd(&sv.hdr->ngen, 1u)] = (int32_t)row;
            };
            // one stage: wait until it is free, describe it, start its copy
            auto put = [&](const StageInfo& info, const unsigned char* src, uint32_t bytes) -> bool {
                const int stage = (int)(g % (uint64_t)nstage);
                if (g >= (uint64_t)nstage) {
                    // wait (bounded) for the scanners to release the stage; stop as soon as the CTA
                    // is dead (its scanners then release nothing more)
                    const uint32_t ph = (uint32_t)(((g / (uint64_t)nstage) - 1) & 1u);
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_wait_bounded(&st.empty[stage], ph, 1000000ull)) {
                        if (*vdead || globaltimer_ns() - t0 > kWaitLimitNs) {
                            *vdead = 1u;
                            return false;
                        }
                    }
                }
                if (*vdead) return false;
                // No proxy fence: the scanners' reads of this stage are ordered before the copy by
                // their arrival on its empty barrier and the wait above, and the description written
                // here reaches them through the full barrier's release (the arrival below).
                st.info[stage] = info;
                mbar_arrive_expect_tx(&st.full[stage], bytes);
                // test hook: CTA 0 withholds the copy of chunk stall_chunk, so that stage never fills
                // and the scanners' bounded wait on it runs out (no copy is left in flight)
                const bool withhold = bytes && blockIdx.x == 0 && a.stall_chunk >= 0 && g == (uint64_t)a.stall_chunk;
                if (withhold)
                    st.withheld = (uint32_t)g + 1u;
                else if (bytes)
                    bulk_g2s(ring + (size_t)stage * chunk_bytes, src, bytes, &st.full[stage]);
                ++g;
                return true;
            };
            // A CTA's first two units are fixed (claims gridDim.x apart), so the ring fills at once
            // and the first claim from the counter -- which waits for the scratch to be cleared --
            // comes a whole unit later.  The next unit is claimed as soon as the current one starts
            // and its parameters are requested after the current unit's second chunk, so both are in
            // flight while the unit is issued (a claim or a parameter read answered at once would
            // leave the ring unfilled at every unit boundary).
            int64_t q = blockIdx.x;
            Unit u = unit_of(a, q < Q ? q : 0);
            RowParams p = load_params(a, u.row);
            while (q < Q && !*vdead) {
                if (a.route == kRouteStream && routed_to_cluster(p.T, p.P, p.MP)) {
                    if (u.seg == 0) list_for_cluster(u.row);
                    q = claim();
                    if (q < Q) {
                        u = unit_of(a, q);
                        p = load_params(a, u.row);
                    }
                    continue;
                }
                st.ulog[nput % kUnitLog] = q;
                ++nput;
                StageInfo info;
                info.row = u.row;
                info.seg = u.seg;
                info.nseg = u.nseg;
                info.p = p;
                const RowGeom geo = row_geom<ES>(a, u.row);
                const UnitGeom ug = unit_geom(geo, u.seg, u.nseg, chunk_bytes);
                const unsigned char* base = reinterpret_cast<const unsigned char*>(geo.a0) + ug.v_lo * 16;
                const uint64_t ubytes = (uint64_t)(ug.v_hi - ug.v_lo) * 16;
                int64_t qn = Q;
                Unit un = u;
                RowParams pn = p;
                const bool claimed = true;
                qn = claim();
                const int c_read = min(1, ug.nchunks - 1);
                for (int c = 0; c < ug.nchunks; ++c) {
                    const uint64_t off = (uint64_t)c * chunk_bytes;
                    const uint32_t bytes = (uint32_t)min((uint64_t)chunk_bytes, ubytes - min(ubytes, off));
                    if (!put(info, base + off, bytes)) break;
                    if (c == c_read && qn < Q) {
                        un = unit_of(a, qn);
                        pn = load_params(a, un.row);
                    }
                }
                if (*vdead) {  // the dead path below starts from the first unit not put in the ring
                    q = claimed ? qn : claim();
                    break;
                }
                q = qn;
                u = un;
                p = pn;
            }
            if (!*vdead) {
                StageInfo end;
                end.row = -1;
                end.seg = 0;
                end.nseg = 1;
                (void)put(end, nullptr, 0);
            }
            st.units_put = nput;
            // A unit claimed but not put in the ring (after a timeout) is settled here: listed for
            // the cluster kernel if it is one of its rows, reported TIMEOUT otherwise.
            auto settle = [&](int64_t qq) {
                const Unit uu = unit_of(a, qq);
                const RowParams pp = load_params(a, uu.row);
                if (a.route == kRouteStream && routed_to_cluster(pp.T, pp.P, pp.MP)) {
                    if (uu.seg == 0) list_for_cluster(uu.row);
                } else {
                    fail_unit(a, sv, qq);
                }
            };
            if (!waited) {
                wait_prerequisite();  // this grid completes after the one it waits for
                waited = true;
            }
            if (*vdead && q < Q) settle(q);
            // A CTA whose wait gave up stops claiming and leaves the rest to the others.  The last CTA
            // to stop claiming settles whatever nobody claimed -- units are left only when CTAs died.
            if (atomicAdd(&sv.hdr->done, 1u) + 1u == gridDim.x) {
                __threadfence();
                for (int64_t qq = claim_counter(); qq < Q; qq = claim_counter()) settle(qq);
            }
            st.issued_lo = (uint32_t)g;
            __threadfence_block();
            *(volatile uint32_t*)&st.producer_done = 1u;
        }
        return;
    }

    // ================= resolver warps =================
    // Resolver r takes units r, r + kResolvers, ... (unit j sits in slot j % kSlots).
    if (warp >= kResolverWarp && warp < kResolverWarp + kResolvers) {
        const uint32_t r = (uint32_t)(warp - kResolverWarp);
        ResolverSpace& rs = st.rs[r];
        auto push = [&](const Task& t) {  // lane 0 only; waits (bounded) for queue space
            const uint64_t t0 = globaltimer_ns();
            while (*(volatile uint32_t*)&rs.q_tail - *(volatile uint32_t*)&rs.q_head >= (uint32_t)kTaskQueue) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    *vdead = 1u;
                    return;
                }
                __nanosleep(200);
            }
            const uint32_t tail = *(volatile uint32_t*)&rs.q_tail;
            rs.q[tail % kTaskQueue] = t;
            __threadfence_block();
            *(volatile uint32_t*)&rs.q_tail = tail + 1;
        };
        wait_prerequisite();  // the scratch (partials, counters) is cleared
        uint32_t j = r;       // the next unit this resolver takes
        for (;; j += kResolvers) {
            const int sl = (int)(j % kSlots);
            RowSlot& slot = st.slot[sl];
            bool ok = mbar_wait_bounded(&st.slot_full[sl], (j / kSlots) & 1u, wait_ns);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                *vdead = 1u;
                break;
            }
            if (slot.row < 0) break;  // no more work
            // take what the unit needs from the slot and free the slot at once
            const Job jb = take_unit(a, rs, slot, *vdead != 0);
            if (lane == 0) {
                slot.lcount = 0;
                slot.runkey = key_neg_inf;
                __threadfence_block();
                mbar_arrive(&st.slot_free[sl]);
            }
            const Task t = (jb.nseg == 1) ? finish_row<TIn>(a, rs, jb) : finish_segment<TIn>(a, sv, rs, jb);
            // hand back what needs the scanners
            __syncwarp();
            if (lane == 0 && t.kind) push(t);
            __syncwarp();
        }
        if (*vdead && lane == 0) {
            // This resolver's units put in the ring but not resolved get a TIMEOUT outcome, once the
            // producer has stopped putting units (bounded wait).
            const uint64_t t0 = globaltimer_ns();
            while (!*(volatile uint32_t*)&st.producer_done && globaltimer_ns() - t0 < 2 * kWaitLimitNs) __nanosleep(1000);
            const uint32_t nput = *(volatile uint32_t*)&st.units_put;
            for (uint32_t k = j; k < nput; k += kResolvers)
                if (nput - k <= (uint32_t)kUnitLog) fail_unit(a, sv, st.ulog[k % kUnitLog]);
        }
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(&st.resolvers_done, 1u);
        }
        return;
    }

    // ================= scanner warps =================
    // Take every queued row (all scanner threads together) until the queue is seen empty.
    auto drain = [&]() {
        for (;;) {
            bool any = false;
            for (int r = 0; r < kResolvers; ++r) {
                ResolverSpace& rs = st.rs[r];
                if (tid == 0) st.q_seen = *(volatile uint32_t*)&rs.q_tail;
                cta_sync();
                const uint32_t tail = st.q_seen, head = rs.q_head;
                cta_sync();
                if (tail == head) continue;
                any = true;
                for (uint32_t h = head; h != tail; ++h) {
                    const Task t = rs.q[h % kTaskQueue];
                    run_task<TIn>(a, s, t);
                    cta_sync();
                }
                if (tid == 0) *(volatile uint32_t*)&rs.q_head = tail;
            }
            if (!any) break;
        }
    };

    uint64_t g = 0;  // chunks consumed, in the producer's order
    uint32_t j = 0;  // units handed over so far
    bool dead = false;
    bool finished = false;
    for (;;) {
        // ---- the next unit: its first stage carries its description
        int stage = (int)(g % (uint64_t)nstage);
        uint32_t parity = (uint32_t)((g / (uint64_t)nstage) & 1u);
        if (!dead && !mbar_wait_bounded(&st.full[stage], parity, wait_ns)) dead = true;
        // one barrier decides whether anything but streaming is due: a timeout (every scanner warp
        // stops at the same unit) or rows queued back by the resolvers
        bool tasks = false;
        if (tid == 0)
            for (int r = 0; r < kResolvers; ++r)
                tasks |= *(volatile uint32_t*)&st.rs[r].q_tail != st.rs[r].q_head;
        if (cta_sync_or((dead || tasks) ? 1 : 0)) {
            if (cta_sync_or(dead ? 1 : 0)) {
                dead = true;
                *vdead = 1u;
                break;
            }
            drain();
        }
        const StageInfo info = st.info[stage];
        if (info.row < 0) {  // no more work
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.empty[stage]);
            ++g;
            finished = true;
            break;
        }
        const int sl = (int)(j % kSlots);
        RowSlot& slot = st.slot[sl];
        if (j >= kSlots && !mbar_wait_bounded(&st.slot_free[sl], ((j / kSlots) - 1) & 1u, wait_ns)) dead = true;
        const int64_t row = info.row;
        const RowParams p = info.p;
        const RowGeom geo = row_geom<ES>(a, row);
        const UnitGeom ug = unit_geom(geo, info.seg, info.nseg, chunk_bytes);
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

        // ragged head (segment 0) and tail (last segment), warp 0 lanes: listed unconditionally at
        // the end of the unit, the resolver filters them
        const int nh = (info.seg == 0) ? geo.nhead : 0;
        const int nt = (info.seg == info.nseg - 1) ? geo.ntail : 0;
        const int nx = nh + nt;
        float xv = -INFINITY;
        int32_t xidx = 0;
        if (tid < nx) {
            xidx = (tid < nh) ? tid : (int32_t)(a.V - geo.ntail + (tid - nh));
            xv = E::load1(geo.rowp, xidx);
        }

        float wrun = -INFINITY;  // this warp's running maximum over the unit (same in all its lanes)
        for (int c = 0; c < ug.nchunks; ++c, ++g) {
            stage = (int)(g % (uint64_t)nstage);
            parity = (uint32_t)((g / (uint64_t)nstage) & 1u);
            const uint64_t off = (uint64_t)c * chunk_bytes;
            const int64_t v0 = ug.v_lo + (int64_t)(off / 16);
            const int nv = (int)min((uint64_t)(chunk_bytes / 16), (uint64_t)(ug.v_hi - v0));
            const uint4* cv = reinterpret_cast<const uint4*>(ring + (size_t)stage * chunk_bytes);
            const int32_t e0 = geo.nhead + (int32_t)(v0 * (16 / ES));
            if (c > 0 && !dead && !mbar_wait_bounded(&st.full[stage], parity, wait_ns)) dead = true;
            dead = __any_sync(0xFFFFFFFFu, dead);
            if (dead && lane == 0) *vdead = 1u;  // the producer stops issuing at once
            if (c == 0) {
                // first chunk: a pass for the maximum alone, published to the slot's running maximum,
                // so the listing pass below tests against the whole chunk's maximum (a warp's own
                // share would list several times more tokens, each through a shared counter).  Every
                // scanner thread reaches the barrier, dead or not.
                if (!dead && nv > 0) {
                    wrun = warp_max_nan(scan_max_list<TIn, false>(cv, nv, e0, INFINITY, nolist));
                    if (lane == 0 && !isnan(wrun)) atomicMax(&slot.runkey, fkey(wrun));
                }
                cta_sync();
            }
            if (!dead && nv > 0) {
                float cm;
                if (c == 0) {
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
            // a stage is released only once scanned: after a timeout its copy may never have landed
            // (or may still land), so it must not be handed back for another copy
            if (lane == 0 && !dead) mbar_arrive(&st.empty[stage]);
        }
        // hand the unit over: ragged elements (listed), this warp's maximum, arrive on the slot
        if (tid < nx) list_token(xv, xidx);
        const float xm = warp_max_nan((tid < nx) ? xv : -INFINITY);
        if (lane == 0) slot.wmax[warp] = dead ? __uint_as_float(0x7FC00000u) : fmax_nan(wrun, xm);
        if (tid == 0) {
            slot.row = row;
            slot.seg = info.seg;
            slot.nseg = info.nseg;
            slot.p = p;
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            mbar_arrive(&st.slot_full[sl]);
        }
        ++j;
    }
    if (finished) {  // tell each resolver there is no more work: an end marker in the next unit it takes
        for (int e = 0; e < kResolvers; ++e, ++j) {
            const int sl = (int)(j % kSlots);
            bool ok = j < kSlots || mbar_wait_bounded(&st.slot_free[sl], ((j / kSlots) - 1) & 1u, wait_ns);
            if (tid == 0) st.slot[sl].row = -1;
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                mbar_arrive(&st.slot_full[sl]);
            }
            if (!ok) *vdead = 1u;
        }
    }
    // keep taking queued rows until the resolvers have finished every unit
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        drain();
        if (tid == 0) st.q_seen = *(volatile uint32_t*)&st.resolvers_done;
        cta_sync();
        const bool rdone = st.q_seen == (uint32_t)kResolvers;
        cta_sync();
        if (rdone) {
            drain();
            break;
        }
        if (globaltimer_ns() - t0 > 4 * kWaitLimitNs) break;  // a resolver wait has already given up
        __nanosleep(500);
    }

    // After a timeout, copies still in flight must land before the shared memory is released (the
    // full limit here, whatever the consumer-side limit was).
    if (tid == 0 && *vdead) {
        const uint64_t t1 = globaltimer_ns();
        while (!*(volatile uint32_t*)&st.producer_done && globaltimer_ns() - t1 < kWaitLimitNs) {
        }
        // the last phase issued on each stage completes only once every copy into it has landed
        const uint64_t issued = st.issued_lo;
        const uint64_t q0 = issued > (uint64_t)nstage ? issued - (uint64_t)nstage : 0;
        for (uint64_t q = q0; q < issued; ++q) {
            if (st.withheld == (uint32_t)q + 1u) continue;  // test hook: no copy was started there
            (void)mbar_wait_bounded(&st.full[q % (uint64_t)nstage], (uint32_t)((q / (uint64_t)nstage) & 1u),
                                    kWaitLimitNs);
        }
    }
    wait_prerequisite();  // this grid completes only after the one it waits for
}

}  // namespace tps
