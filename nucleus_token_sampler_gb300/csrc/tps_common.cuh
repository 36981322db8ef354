// tps_common.cuh -- pieces shared by the two row samplers (the cluster kernel and the streaming
// kernel): shared-memory state, block reductions, the sources a pass reads (a slice in shared
// memory or a whole row in global memory), the cluster/single-CTA "topology" the exchanges use,
// histogram-located cuts with exact refinement, candidate resolution and the exponential race.
//
// The chain is the one on "What do temperature, top-k and top-p each do to the next-token
// distribution, and in what order does a serving engine apply them?" ('A strong answer'), with
// the top-p rule of "Implement batched top-p sampling with temperature" ('How to approach it').
#pragma once

#include <cooperative_groups.h>
#include <cfloat>

#include "tps_device.cuh"

namespace tps {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;            // level-1 bins over d, width 1/8 (last bin: d >= 31.875)
constexpr float kBinScale = 8.f;
constexpr int kSubBins = 256;         // sub-bins over a key interval
constexpr int kCand = 256;            // candidates resolved by sorting, per CTA and per cluster
constexpr int kMaxExtra = 16;         // ragged head/tail elements fetched with plain loads
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s bound on every wait

enum RowStatus : int32_t { kRowOk = 0, kRowNan = 1, kRowAllMasked = 2, kRowBadParam = 3, kRowTimeout = 4 };

struct Args {
    const void* logits;
    int64_t B, V, ld;
    const float* temperature;
    const int32_t* top_k;
    const float* top_p;
    const float* min_p;
    const uint64_t* seed;
    uint64_t step;
    int32_t* out_token;
    float* out_probs;
    int32_t* out_status;
    float* out_cutoff;
    int32_t* out_kept;
    uint32_t slice_cap;  // bytes reserved for the slice at the start of dynamic shared memory
};

struct Shared {
    uint64_t mbar;
    // --- values the other CTAs of the cluster read through distributed shared memory
    float pub_max;
    uint32_t pub_timeout;
    uint32_t pub_minidx;
    uint32_t pub_nsurv;
    uint32_t pub_minkey;
    uint32_t pub_gcnt;
    uint32_t pub_gkmin;
    uint32_t pub_gkmax;
    double pub_k64;
    int32_t pub_idx;
    // --- ragged elements
    int32_t nx;
    float xz[kMaxExtra];
    int32_t xi[kMaxExtra];
    // --- block reduction scratch and broadcast slots
    float rf[kWarps];
    uint32_t ra[kWarps];
    uint32_t rb[kWarps];
    uint64_t r64[kWarps];
    ArgBest rab[kWarps];
    uint32_t bu[8];
    uint64_t b64[4];
    float bf[2];
    ArgBest bab;
    // --- gather bookkeeping: offset and count of each CTA's list
    uint32_t goff[16];
    uint32_t gcnt[16];
    uint32_t gtotal;
    // --- histogram: local, then (after the cluster reduction) the full reduced histogram
    uint32_t hcnt[kBins];
    uint64_t hmass[kBins];
    union alignas(16) {
        struct {  // this CTA's share of the reduced histogram (read by the other CTAs)
            uint32_t rcnt[kBins];
            uint64_t rmass[kBins];
        } sh;
        struct {  // gathered candidates (key << 32 | ~index), sorted descending, and mass prefixes
            uint64_t sbuf[kCand];
            uint64_t pre[kCand + 1];
        } cd;
    } u;
    // --- this CTA's candidate list (read by the other CTAs)
    uint32_t ncand;
    uint32_t ckey[kCand];
    uint32_t cidx[kCand];
};

// ---------------------------------------------------------------------------------------------
// CTA barriers over the kThreads sampling threads only (named barrier 1).  The streaming kernel
// adds one producer warp that never joins them; in the cluster kernel they cover the whole CTA.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void cta_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ int cta_sync_or(int pred)
{
    int r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.s32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, %2, pi;\n\t"
        "selp.s32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred), "n"(kThreads)
        : "memory");
    return r;
}

__device__ __forceinline__ int cta_sync_count(int pred)
{
    int r;
    asm volatile(
        "{\n\t.reg .pred pi;\n\t"
        "setp.ne.s32 pi, %1, 0;\n\t"
        "bar.red.popc.u32 %0, 1, %2, pi;\n\t}"
        : "=r"(r)
        : "r"(pred), "n"(kThreads)
        : "memory");
    return r;
}

// ---------------------------------------------------------------------------------------------
// Block-level helpers (every thread of the CTA must call them).  Each starts with a barrier so
// its scratch can be reused right after the previous call.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, Shared& s)
{
    v = warp_sum_u32(v);
    cta_sync();
    if ((threadIdx.x & 31) == 0) s.ra[threadIdx.x >> 5] = v;
    cta_sync();
    uint32_t r = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) r += s.ra[w];
    return r;
}

__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, Shared& s)
{
    v = warp_min_u32(v);
    cta_sync();
    if ((threadIdx.x & 31) == 0) s.rb[threadIdx.x >> 5] = v;
    cta_sync();
    uint32_t r = s.rb[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = min(r, s.rb[w]);
    return r;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, Shared& s)
{
    v = warp_max_u32(v);
    cta_sync();
    if ((threadIdx.x & 31) == 0) s.rb[threadIdx.x >> 5] = v;
    cta_sync();
    uint32_t r = s.rb[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = max(r, s.rb[w]);
    return r;
}

__device__ __forceinline__ ArgBest block_argbest(ArgBest a, Shared& s)
{
    a = warp_argbest(a);
    cta_sync();
    if ((threadIdx.x & 31) == 0) s.rab[threadIdx.x >> 5] = a;
    cta_sync();
    ArgBest r = s.rab[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w)
        if (better(s.rab[w].key, s.rab[w].idx, r.key, r.idx)) r = s.rab[w];
    return r;
}

// Exclusive scan of one u64 per thread; returns the prefix, writes the total to *total.
__device__ __forceinline__ uint64_t block_exscan_u64(uint64_t v, Shared& s, uint64_t* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    cta_sync();
    if (lane == 31) s.r64[warp] = x;
    cta_sync();
    uint64_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint64_t t = s.r64[w];
        if (w < warp) before += t;
        all += t;
    }
    *total = all;
    return before + x - v;
}

// ---------------------------------------------------------------------------------------------
// Topologies: the CTAs that share one row.  ClusterTopo is a thread-block cluster exchanging
// through distributed shared memory; SoloTopo is a single CTA (map() is the identity).
// ---------------------------------------------------------------------------------------------
struct ClusterTopo {
    cg::cluster_group g;
    uint32_t C, rank;
    __device__ __forceinline__ ClusterTopo() : g(cg::this_cluster())
    {
        C = g.num_blocks();
        rank = g.block_rank();
    }
    __device__ __forceinline__ void sync() { g.sync(); }
    template <typename T>
    __device__ __forceinline__ T* map(T* p, uint32_t r)
    {
        return g.map_shared_rank(p, r);
    }
};

struct SoloTopo {
    uint32_t C = 1, rank = 0;
    __device__ __forceinline__ void sync() { cta_sync(); }
    template <typename T>
    __device__ __forceinline__ T* map(T* p, uint32_t)
    {
        return p;
    }
};

// ---------------------------------------------------------------------------------------------
// Sources: what one pass reads.  Both apply f(z, i) to every element they cover -- 16-byte vectors
// (four loaded before any is processed, so the latency overlaps even when f holds atomics), then
// the ragged head/tail elements kept in s.xz/s.xi.
// ---------------------------------------------------------------------------------------------
template <typename TIn, bool kGlobal>
struct VecSource {
    const uint4* vec;  // kGlobal: the row's aligned interior in global memory; else a shared slice
    int nvec;
    int64_t elem0;     // row index of the first element of vec[0]

    __device__ __forceinline__ uint4 load(int v) const
    {
        if constexpr (kGlobal) return __ldg(vec + v);
        else return vec[v];
    }

    template <typename F>
    __device__ __forceinline__ void for_each(const Shared& s, F&& f) const
    {
        using E = Elem<TIn>;
        constexpr int U = 4;
        int v = threadIdx.x;
        for (; v + (U - 1) * kThreads < nvec; v += U * kThreads) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) w[u] = load(v + u * kThreads);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float z[E::kPerVec];
                E::unpack(w[u], z);
                const int32_t i0 = (int32_t)elem0 + (v + u * kThreads) * E::kPerVec;
#pragma unroll
                for (int j = 0; j < E::kPerVec; ++j) f(z[j], i0 + j);
            }
        }
        for (; v < nvec; v += kThreads) {
            float z[E::kPerVec];
            E::unpack(load(v), z);
            const int32_t i0 = (int32_t)elem0 + v * E::kPerVec;
#pragma unroll
            for (int j = 0; j < E::kPerVec; ++j) f(z[j], i0 + j);
        }
        for (int x = threadIdx.x; x < s.nx; x += kThreads) f(s.xz[x], s.xi[x]);
    }
};
template <typename TIn>
using Slice = VecSource<TIn, false>;
template <typename TIn>
using GlobalRow = VecSource<TIn, true>;

// Maximum (NaN-propagating) over nvec 16-byte vectors, listing every element above thr through
// list(z, i).  Each thread takes 16 elements per step and reduces them with a tree of max
// operations; only a step whose maximum exceeds thr is looked at element by element, so a pass
// costs about one instruction per element when little is listed.
template <typename TIn, bool kGlobal, typename ListF>
__device__ __forceinline__ float scan_max_list(const uint4* vec, int nvec, int32_t elem0, float thr, ListF&& list)
{
    using E = Elem<TIn>;
    constexpr int EPV = E::kPerVec;
    constexpr int U = 16 / EPV;  // vectors per step
    const uint4 neg_inf = (EPV == 4) ? make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u)
                                     : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    float cm = -INFINITY;
    for (int v = threadIdx.x; v < nvec; v += U * kThreads) {
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vi = v + u * kThreads;
            if (vi < nvec) {
                if constexpr (kGlobal) w[u] = __ldg(vec + vi);
                else w[u] = vec[vi];
            } else {
                w[u] = neg_inf;
            }
        }
        float z[U * EPV];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float t[EPV];
            E::unpack(w[u], t);
#pragma unroll
            for (int j = 0; j < EPV; ++j) z[u * EPV + j] = t[j];
        }
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = fmax_nan(z[j], z[j + 8]);
#pragma unroll
        for (int j = 0; j < 4; ++j) m8[j] = fmax_nan(m8[j], m8[j + 4]);
        const float m = fmax_nan(fmax_nan(m8[0], m8[2]), fmax_nan(m8[1], m8[3]));
        cm = fmax_nan(cm, m);
        if (m > thr) {
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < EPV; ++j)
                    if (z[u * EPV + j] > thr) list(z[u * EPV + j], elem0 + (v + u * kThreads) * EPV + j);
        }
    }
    return cm;
}

// A listing threshold that min-p, measured against any maximum >= m, surely rejects at or below:
// m - (L_hi T (1 + 1e-5) + |m| 2^-20).  The margins cover the float rounding of this expression
// and of d = (zmax - z) / T, so every token at or below it has d > L_hi against the true maximum.
__device__ __forceinline__ float list_threshold(float m, float lt_hi)
{
    return m - (lt_hi + fabsf(m) * 0x1p-20f);
}

__device__ __forceinline__ int bin_of(float d)
{
    return min(__float2int_rz(d * kBinScale), kBins - 1);
}

// Cluster-wide sum of the local histogram hcnt/hmass[0, nb) into hcnt/hmass of every CTA.
// Step 1: CTA c sums its share of the bins over all CTAs (one remote read per thread) into
// u.sh; step 2: every CTA copies all shares back into its own hcnt/hmass.
template <typename Topo>
__device__ __forceinline__ void cluster_reduce_hist(Topo& topo, Shared& s, int nb)
{
    const uint32_t C = topo.C, rank = topo.rank;
    if (C == 1) {  // a single CTA already holds the full histogram
        cta_sync();
        return;
    }
    const int per = (nb + (int)C - 1) / (int)C;
    const int b0 = min(nb, (int)rank * per), b1 = min(nb, b0 + per);
    topo.sync();  // every local histogram complete; nobody reads my previous share any more
    for (int b = b0 + (int)threadIdx.x; b < b1; b += kThreads) {
        s.u.sh.rcnt[b] = 0;
        s.u.sh.rmass[b] = 0;
    }
    cta_sync();
    const int npairs = (b1 - b0) * (int)C;
    for (int p = threadIdx.x; p < npairs; p += kThreads) {
        const int b = b0 + p / (int)C;
        const uint32_t r = (uint32_t)(p % (int)C);
        const uint32_t c = *topo.map(&s.hcnt[b], r);
        if (c) {
            atomicAdd(&s.u.sh.rcnt[b], c);
            atomicAdd((unsigned long long*)&s.u.sh.rmass[b],
                      (unsigned long long)*topo.map(&s.hmass[b], r));
        }
    }
    topo.sync();  // all shares complete; nobody reads another CTA's hcnt/hmass any more
    for (int b = threadIdx.x; b < nb; b += kThreads) {
        const uint32_t owner = (uint32_t)(b / per);
        s.hcnt[b] = *topo.map(&s.u.sh.rcnt[b], owner);
        s.hmass[b] = *topo.map(&s.u.sh.rmass[b], owner);
    }
    cta_sync();
}

struct Sel {
    uint32_t key;    // the lowest kept class (its logit's key)
    uint64_t cnt;    // tokens kept, counting from the top
    uint64_t mass;   // their fixed-point mass
};

struct Crit {
    bool by_mass;     // false: keep a class while (count above it) < tcnt
    uint64_t tcnt;    // true:  keep a class while (mass above it) < tmass
    double tmass;
    __device__ __forceinline__ bool keep(uint64_t cnt_above, uint64_t mass_above) const
    {
        return by_mass ? ((double)mass_above < tmass) : (cnt_above < tcnt);
    }
};

// Scan the (full) histogram hcnt/hmass[0, nb) from bin 0 (largest logits) down and return the
// last non-empty bin whose (count, mass) above satisfies the criterion.  nb <= kThreads.
__device__ __forceinline__ void scan_bins(Shared& s, int nb, const Crit& cr, uint64_t C0, uint64_t A0,
                                          int* out_bin, uint64_t* out_c, uint64_t* out_a)
{
    const int b = threadIdx.x;
    const uint64_t c = (b < nb) ? s.hcnt[b] : 0;
    const uint64_t m = (b < nb) ? s.hmass[b] : 0;
    uint64_t tot;
    const uint64_t cpre = block_exscan_u64(c, s, &tot);
    const uint64_t mpre = block_exscan_u64(m, s, &tot);
    const uint32_t best = (c > 0 && cr.keep(C0 + cpre, A0 + mpre)) ? (uint32_t)b + 1u : 0u;
    const uint32_t bb = block_max_u32(best, s);
    if (bb != 0 && b == (int)bb - 1) {
        s.b64[0] = C0 + cpre;
        s.b64[1] = A0 + mpre;
    }
    cta_sync();
    *out_bin = (int)bb - 1;
    *out_c = bb ? s.b64[0] : C0;
    *out_a = bb ? s.b64[1] : A0;
    cta_sync();
}

// Sort u.cd.sbuf[0, n) (n <= kThreads, distinct values) descending: thread t counts the entries
// larger than its own (broadcast reads, two at a time) and scatters it to that rank.  Two barriers
// instead of a bitonic network's log^2 n.
__device__ __forceinline__ void block_sort_desc(Shared& s, int n)
{
    uint64_t* sb = s.u.cd.sbuf;
    uint64_t* tmp = s.u.cd.pre;  // kCand + 1 entries of scratch
    const int t = threadIdx.x;
    uint64_t v = 0;
    int rank = 0;
    if (t < n) {
        v = sb[t];
        int j = 0;
        for (; j + 1 < n; j += 2) {
            const ulonglong2 w = *reinterpret_cast<const ulonglong2*>(sb + j);
            rank += (w.x > v) + (w.y > v);
        }
        if (j < n) rank += (sb[j] > v);
    }
    cta_sync();
    if (t < n) tmp[rank] = v;
    cta_sync();
    if (t < n) sb[t] = tmp[t];
    cta_sync();
}

__device__ __forceinline__ uint32_t sb_key(uint64_t v) { return (uint32_t)(v >> 32); }
__device__ __forceinline__ int32_t sb_idx(uint64_t v) { return (int32_t)(~(uint32_t)v); }
__device__ __forceinline__ uint64_t sb_make(uint32_t key, uint32_t idx)
{
    return ((uint64_t)key << 32) | (uint64_t)(~idx);
}

// Fill u.cd.pre[0, n] with the exclusive prefix of the fixed-point masses of sbuf[0, n).
__device__ __forceinline__ void prefix_masses(Shared& s, const RowCtx& r, int n)
{
    const int t = threadIdx.x;  // n <= kCand == kThreads
    const uint64_t q = (t < n) ? qmass_d(dist(r, key_to_float(sb_key(s.u.cd.sbuf[t])))) : 0;
    uint64_t tot;
    const uint64_t run = block_exscan_u64(q, s, &tot);
    if (t < n) s.u.cd.pre[t] = run;
    if (t == 0) s.u.cd.pre[n] = tot;
    cta_sync();
}

// Walk the classes of the sorted candidates sbuf[0, n) and return the last class whose
// (count, mass) above -- offset by (C0, A0) -- satisfies the criterion.
__device__ __forceinline__ Sel walk_classes(Shared& s, int n, const Crit& cr, uint64_t C0, uint64_t A0)
{
    const uint64_t* sb = s.u.cd.sbuf;
    const int t = threadIdx.x;
    bool start = false;
    if (t < n) {
        start = (t == 0) || sb_key(sb[t - 1]) != sb_key(sb[t]);
    }
    const uint32_t best = (start && cr.keep(C0 + (uint64_t)t, A0 + s.u.cd.pre[t])) ? (uint32_t)t + 1u : 0u;
    const uint32_t sbst = block_max_u32(best, s);
    const int st = sbst ? (int)sbst - 1 : 0;
    const uint32_t end = (start && t > st) ? (uint32_t)t : (uint32_t)n;
    const uint32_t e = block_min_u32(end, s);
    Sel out;
    out.key = sb_key(sb[st]);
    out.cnt = C0 + e;
    out.mass = A0 + s.u.cd.pre[e];
    cta_sync();
    return out;
}

// Copy every CTA's candidate list (counts in pub_gcnt) into u.cd.sbuf and sort it.  Returns n.
template <typename Topo>
__device__ __forceinline__ int gather_and_sort(Topo& topo, Shared& s)
{
    const uint32_t C = topo.C;
    if (threadIdx.x < 32) {  // lane r reads rank r's count; exclusive prefix over the ranks
        const uint32_t lane = threadIdx.x;
        const uint32_t cnt = (lane < C) ? *topo.map(&s.pub_gcnt, lane) : 0u;
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
        if (lane == 31) s.gtotal = inc;
    }
    cta_sync();
    const uint32_t n = s.gtotal;
    for (uint32_t rr = 0; rr < C; ++rr) {  // each count <= kCand == kThreads
        const uint32_t off = s.goff[rr], cnt = s.gcnt[rr];
        if (threadIdx.x < cnt) {
            const uint32_t k = *topo.map(&s.ckey[threadIdx.x], rr);
            const uint32_t i = *topo.map(&s.cidx[threadIdx.x], rr);
            s.u.cd.sbuf[off + threadIdx.x] = sb_make(k, i);
        }
    }
    cta_sync();
    block_sort_desc(s, (int)n);
    return (int)n;
}

// Race key in float (for pruning) and in double (for the decision) of kept token i.
struct RaceCtx {
    uint32_t k0, k1;    // Philox key = seed
    uint32_t row, s_lo, s_hi;
};

__device__ __forceinline__ float race_u(const RaceCtx& rc, int32_t i)
{
    const uint4 x = philox4x32_10(make_uint4((uint32_t)i >> 2, rc.row, rc.s_lo, rc.s_hi), rc.k0, rc.k1);
    return (float)uniform_grid(pick_word(x, (uint32_t)i & 3u)) * 0x1p-24f;
}

__device__ __forceinline__ float race_key32(float d, float u) { return -d - logf(-logf(u)); }

__device__ __forceinline__ double race_key64(const RowCtx& r, float z, float u)
{
    const double d = __ddiv_rn(__dsub_rn((double)r.zmax, (double)z), (double)r.T);
    const double g = log(-log((double)u));
    return __dsub_rn(-d, g);
}

// Margin between the float race key and the double one (both tokens' errors), for a row whose
// kept tokens have d <= dcut.
__device__ __forceinline__ float race_tol(float dcut) { return 1e-5f + 1e-6f * dcut; }

// Refine the cut inside level-1 bin `bin` (tokens with key >= key_lo that survive min-p), given
// the (count, mass) of the survivors above the bin.  Exact: ends with a sorted candidate list or
// with a single logit value.
template <typename Topo, typename Src>
__device__ Sel refine_bin(Topo& topo, Shared& s, const Src& sl, const RowCtx& r, float zc, int bin, uint32_t key_lo,
                          const Crit& cr, uint64_t C0, uint64_t A0)
{
    const uint32_t C = topo.C;
    uint32_t klo = 0, khi = 0xFFFFFFFFu;
    bool by_bin = true;
    for (int iter = 0; iter < 8; ++iter) {
        // Gather the tokens of the current range (a level-1 bin, or a key interval).
        topo.sync();  // nobody still reads my candidate list, published counts or shares
        if (threadIdx.x == 0) s.ncand = 0;
        cta_sync();
        uint32_t lcnt = 0, lmin = 0xFFFFFFFFu, lmax = 0;
        const uint32_t lo = klo, hi = khi;
        sl.for_each(s, [&](float z, int32_t i) {
            if (!(z > zc)) return;
            const uint32_t key = fkey(z);
            if (key < key_lo || key < lo || key > hi) return;
            const float d = dist(r, z);
            if (by_bin && bin_of(d) != bin) return;
            if (!minp_ok(r, z, d)) return;
            ++lcnt;
            lmin = min(lmin, key);
            lmax = max(lmax, key);
            if (*(volatile uint32_t*)&s.ncand < (uint32_t)kCand) {
                const uint32_t slot = atomicAdd(&s.ncand, 1u);
                if (slot < (uint32_t)kCand) {
                    s.ckey[slot] = key;
                    s.cidx[slot] = (uint32_t)i;
                }
            }
        });
        const uint32_t cnt = block_sum_u32(lcnt, s);
        const uint32_t kmn = block_min_u32(lmin, s);
        const uint32_t kmx = block_max_u32(lmax, s);
        if (threadIdx.x == 0) {
            s.pub_gcnt = min(cnt, (uint32_t)kCand);
            s.pub_nsurv = cnt;
            s.pub_gkmin = kmn;
            s.pub_gkmax = kmx;
        }
        topo.sync();
        if (threadIdx.x < 32) {
            const uint32_t lane = threadIdx.x;
            uint32_t tc = 0, gmn = 0xFFFFFFFFu, gmx = 0;
            if (lane < C) {
                tc = *topo.map(&s.pub_nsurv, lane);
                gmn = *topo.map(&s.pub_gkmin, lane);
                gmx = *topo.map(&s.pub_gkmax, lane);
            }
            tc = warp_sum_u32(tc);
            gmn = warp_min_u32(gmn);
            gmx = warp_max_u32(gmx);
            if (lane == 0) {
                s.bu[4] = tc;
                s.bu[5] = gmn;
                s.bu[6] = gmx;
            }
        }
        cta_sync();
        const uint64_t total = s.bu[4];
        const uint32_t gmin = s.bu[5], gmax = s.bu[6];
        if (total == 0) {  // cannot happen for a bin chosen as non-empty; keep a valid answer
            Sel o;
            o.key = key_lo;
            o.cnt = C0;
            o.mass = A0;
            return o;
        }
        if (gmin == gmax) {  // a single logit value: one class
            const uint64_t q = qmass_d(dist(r, key_to_float(gmin)));
            Sel o;
            o.key = gmin;
            o.cnt = C0 + total;
            o.mass = A0 + total * q;
            return o;
        }
        if (total <= (uint64_t)kCand) {
            const int n = gather_and_sort(topo, s);
            prefix_masses(s, r, n);
            return walk_classes(s, n, cr, C0, A0);
        }
        // Too many: split the key range [gmin, gmax] into sub-bins (sub-bin 0 = largest keys).
        klo = gmin;
        khi = gmax;
        by_bin = false;
        int sh = 0;
        while (((uint64_t)(khi - klo) >> sh) >= (uint64_t)kSubBins) ++sh;
        const int nsub = (int)((uint64_t)(khi - klo) >> sh) + 1;
        for (int b = threadIdx.x; b < kSubBins; b += kThreads) {
            s.hcnt[b] = 0;
            s.hmass[b] = 0;
        }
        cta_sync();
        const uint32_t lo2 = klo, hi2 = khi;
        sl.for_each(s, [&](float z, int32_t) {
            if (!(z > zc)) return;
            const uint32_t key = fkey(z);
            if (key < key_lo || key < lo2 || key > hi2) return;
            const float d = dist(r, z);
            if (!minp_ok(r, z, d)) return;
            const int sb = (int)((hi2 - key) >> sh);
            atomicAdd(&s.hcnt[sb], 1u);
            atomicAdd((unsigned long long*)&s.hmass[sb], (unsigned long long)qmass_d(d));
        });
        cluster_reduce_hist(topo, s, kSubBins);
        int jb;
        uint64_t c_at, a_at;
        scan_bins(s, nsub, cr, C0, A0, &jb, &c_at, &a_at);
        if (jb < 0) jb = 0;
        C0 = c_at;
        A0 = a_at;
        const uint64_t top = (uint64_t)hi2 - ((uint64_t)jb << sh);
        const uint64_t width = (uint64_t)1 << sh;
        const uint64_t bot = (top + 1 >= width) ? top + 1 - width : 0;
        khi = (uint32_t)top;
        klo = (uint32_t)max((uint64_t)lo2, bot);
    }
    // Unreachable in practice (each split shrinks the 32-bit range by 2^8); keep a valid answer.
    Sel o;
    o.key = khi;
    o.cnt = C0;
    o.mass = A0;
    return o;
}

// ---------------------------------------------------------------------------------------------
// Exponential race, decided exactly.  Float keys rank the kept tokens; when the best float key
// leads every other by more than the float/double error margin, it is the double-precision argmax
// too.  Only near-ties (two keys within the margin) are re-evaluated in double precision, exactly
// as the float64 definition computes them, with the lowest index winning equal keys.
// ---------------------------------------------------------------------------------------------
struct WarpResult {
    uint32_t key_cut;
    uint32_t nk;
    uint64_t zk;
    int32_t token;
};

// Resolve a row whose survivors are buf[0, n) (n <= 32, unsorted) with one warp.  Every lane
// returns the same result.
__device__ __forceinline__ WarpResult warp_resolve(const uint64_t* buf, const RowCtx& r, const RaceCtx& rc, uint32_t n,
                                                   bool topk_on, int32_t K, float P)
{
    const uint32_t lane = threadIdx.x & 31;
    uint64_t v = (lane < n) ? buf[lane] : 0;
    // bitonic sort across the warp, descending
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            const bool take_max = ((lane & k2) == 0) == ((lane & j) == 0);
            v = take_max ? (v > o ? v : o) : (v < o ? v : o);
        }
    }
    const uint32_t key = sb_key(v);
    const int32_t idx = sb_idx(v);
    const bool valid = lane < n;
    const float z = key_to_float(key);
    const float d = dist(r, z);
    const uint64_t q = valid ? qmass_d(d) : 0;
    uint64_t inc = q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if ((int)lane >= o) inc += y;
    }
    const uint64_t exc = inc - q;
    const uint64_t total = __shfl_sync(0xFFFFFFFFu, inc, 31);
    const uint32_t prev_key = __shfl_up_sync(0xFFFFFFFFu, key, 1);
    const bool start = valid && (lane == 0 || prev_key != key);
    auto prefix_at = [&](uint32_t e) -> uint64_t {
        const uint64_t x = __shfl_sync(0xFFFFFFFFu, exc, e & 31u);
        return e >= 32 ? total : x;
    };
    // last class start in [0, lim) satisfying the criterion, and the end of that class
    auto cut = [&](uint32_t lim, bool by_mass, uint64_t tcnt, double tmass, uint32_t* st_out, uint32_t* e_out) {
        const bool ok = start && lane < lim && (by_mass ? ((double)exc < tmass) : ((uint64_t)lane < tcnt));
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, ok);
        const uint32_t st = m ? 31u - __clz(m) : 0u;
        const uint32_t ends = __ballot_sync(0xFFFFFFFFu, start && lane < lim && lane > st);
        *st_out = st;
        *e_out = ends ? (uint32_t)(__ffs(ends) - 1) : lim;
    };
    uint32_t ns = n;
    uint64_t zs = total;
    if (topk_on && n > (uint32_t)K) {
        uint32_t st, e;
        cut(n, false, (uint64_t)K, 0.0, &st, &e);
        ns = e;
        zs = prefix_at(e);
    }
    uint32_t nk = ns;
    uint64_t zk = zs;
    if (P < 1.f) {
        uint32_t st, e;
        cut(ns, P > 0.f, 1, (double)P * (double)zs, &st, &e);
        nk = e;
        zk = prefix_at(e);
    }
    const uint32_t key_cut = __shfl_sync(0xFFFFFFFFu, key, (nk - 1) & 31u);
    // race over lanes < nk
    const bool kept = lane < nk;
    float u = 0.f, k32 = -INFINITY;
    if (kept) {
        u = race_u(rc, idx);
        k32 = race_key32(d, u);
    }
    float m32 = k32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m32 = fmaxf(m32, __shfl_xor_sync(0xFFFFFFFFu, m32, o));
    const float tol = race_tol(dist(r, key_to_float(key_cut)));
    const bool fin = kept && k32 >= m32 - tol;
    const uint32_t fm = __ballot_sync(0xFFFFFFFFu, fin);
    int32_t token;
    if (__popc(fm) == 1) {
        token = __shfl_sync(0xFFFFFFFFu, idx, __ffs(fm) - 1);
    } else {
        ArgBest a;
        a.key = -INFINITY;
        a.idx = 0x7FFFFFFF;
        if (fin) {
            a.key = race_key64(r, z, u);
            a.idx = idx;
        }
        token = warp_argbest(a).idx;
    }
    WarpResult res;
    res.key_cut = key_cut;
    res.nk = nk;
    res.zk = zk;
    res.token = token;
    return res;
}

// Resolve a row whose survivors are buf[0, n) (32 < n <= 256, distinct, any order) with one warp:
// rank sort into sorted[], fixed-point mass prefixes in pre[0, n], the top-k and top-p class cuts,
// then the race.  Lane l owns sorted positions [8 l, 8 l + 8).  Every lane returns the same result.
__device__ __forceinline__ WarpResult warp_resolve_big(const uint64_t* buf, uint64_t* sorted, uint64_t* pre, uint32_t n,
                                                       const RowCtx& r, const RaceCtx& rc, bool topk_on, int32_t K,
                                                       float P)
{
    const uint32_t lane = threadIdx.x & 31;
    // rank sort: every entry counts the entries larger than itself
#pragma unroll 1
    for (uint32_t e = lane; e < n; e += 32) {
        const uint64_t v = buf[e];
        uint32_t rank = 0, j = 0;
        for (; j + 1 < n; j += 2) {
            const ulonglong2 w = *reinterpret_cast<const ulonglong2*>(buf + j);
            rank += (w.x > v) + (w.y > v);
        }
        if (j < n) rank += (buf[j] > v);
        sorted[rank] = v;
    }
    __syncwarp();
    const uint32_t p0 = 8 * lane;
    uint64_t q[8];
    uint32_t kk[8];
    uint64_t loc = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t pos = p0 + m;
        kk[m] = (pos < n) ? sb_key(sorted[pos]) : 0u;
        q[m] = (pos < n) ? qmass_d(dist(r, key_to_float(kk[m]))) : 0;
        loc += q[m];
    }
    uint64_t inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if ((int)lane >= o) inc += y;
    }
    uint64_t run = inc - loc;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        if (p0 + m < n) pre[p0 + m] = run;
        run += q[m];
    }
    if (lane == 31) pre[n] = inc;
    __syncwarp();
    const uint32_t prevk = __shfl_up_sync(0xFFFFFFFFu, kk[7], 1);
    bool start[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t pos = p0 + m;
        const uint32_t before = (m == 0) ? prevk : kk[m - 1];
        start[m] = (pos < n) && (pos == 0 || before != kk[m]);
    }
    // last class start in [0, lim) satisfying the criterion, and the end of that class
    auto cut = [&](uint32_t lim, bool by_mass, uint64_t tcnt, double tmass, uint32_t* st_out, uint32_t* e_out) {
        uint32_t best = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t pos = p0 + m;
            if (start[m] && pos < lim && (by_mass ? ((double)pre[pos] < tmass) : ((uint64_t)pos < tcnt)))
                best = pos + 1;
        }
        const uint32_t st = __reduce_max_sync(0xFFFFFFFFu, best);
        const uint32_t s0 = st ? st - 1 : 0;
        uint32_t end = lim;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t pos = p0 + m;
            if (start[m] && pos < lim && pos > s0) end = min(end, pos);
        }
        *st_out = s0;
        *e_out = __reduce_min_sync(0xFFFFFFFFu, end);
    };
    uint32_t ns = n;
    uint64_t zs = pre[n];
    if (topk_on && n > (uint32_t)K) {
        uint32_t st, e;
        cut(n, false, (uint64_t)K, 0.0, &st, &e);
        ns = e;
        zs = pre[e];
    }
    uint32_t nk = ns;
    uint64_t zk = zs;
    if (P < 1.f) {
        uint32_t st, e;
        cut(ns, P > 0.f, 1, (double)P * (double)zs, &st, &e);
        nk = e;
        zk = pre[e];
    }
    const uint32_t key_cut = sb_key(sorted[nk - 1]);
    // race over positions < nk
    float k32[8], uu[8];
    float m32 = -INFINITY;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t pos = p0 + m;
        k32[m] = -INFINITY;
        uu[m] = 0.f;
        if (pos < nk) {
            uu[m] = race_u(rc, sb_idx(sorted[pos]));
            k32[m] = race_key32(dist(r, key_to_float(kk[m])), uu[m]);
            m32 = fmaxf(m32, k32[m]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m32 = fmaxf(m32, __shfl_xor_sync(0xFFFFFFFFu, m32, o));
    const float tol = race_tol(dist(r, key_to_float(key_cut)));
    uint32_t nf = 0, fpos = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m)
        if (p0 + m < nk && k32[m] >= m32 - tol) {
            ++nf;
            fpos = p0 + m;
        }
    const uint32_t nfin = __reduce_add_sync(0xFFFFFFFFu, nf);
    int32_t token;
    if (nfin == 1) {
        const uint32_t who = __ballot_sync(0xFFFFFFFFu, nf != 0);
        token = sb_idx(sorted[__shfl_sync(0xFFFFFFFFu, fpos, __ffs(who) - 1)]);
    } else {
        ArgBest a;
        a.key = -INFINITY;
        a.idx = 0x7FFFFFFF;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t pos = p0 + m;
            if (pos < nk && k32[m] >= m32 - tol) {
                const double k64 = race_key64(r, key_to_float(kk[m]), uu[m]);
                const int32_t i = sb_idx(sorted[pos]);
                if (better(k64, i, a.key, a.idx)) {
                    a.key = k64;
                    a.idx = i;
                }
            }
        }
        token = warp_argbest(a).idx;
    }
    WarpResult res;
    res.key_cut = key_cut;
    res.nk = nk;
    res.zk = zk;
    res.token = token;
    return res;
}

// Best and second-best float race keys (and the best's index) over a set of tokens.
struct Top2 {
    float k1, k2;
    int32_t i1;
    __device__ __forceinline__ void init()
    {
        k1 = k2 = -INFINITY;
        i1 = 0x7FFFFFFF;
    }
    __device__ __forceinline__ void add(float k, int32_t i)
    {
        if (k > k1 || (k == k1 && (uint32_t)i < (uint32_t)i1)) {
            k2 = k1;
            k1 = k;
            i1 = i;
        } else if (k > k2) {
            k2 = k;
        }
    }
    __device__ __forceinline__ void merge(const Top2& o)
    {
        if (o.k1 > k1 || (o.k1 == k1 && (uint32_t)o.i1 < (uint32_t)i1)) {
            k2 = fmaxf(k1, o.k2);
            k1 = o.k1;
            i1 = o.i1;
        } else {
            k2 = fmaxf(k2, o.k1);
        }
    }
};

__device__ __forceinline__ Top2 warp_top2(Top2 t)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Top2 x;
        x.k1 = __shfl_xor_sync(0xFFFFFFFFu, t.k1, o);
        x.k2 = __shfl_xor_sync(0xFFFFFFFFu, t.k2, o);
        x.i1 = __shfl_xor_sync(0xFFFFFFFFu, t.i1, o);
        t.merge(x);
    }
    return t;
}

// ---------------------------------------------------------------------------------------------
// Row-level building blocks used by both kernels.  All threads of the CTA call them.
// ---------------------------------------------------------------------------------------------
struct RowResult {
    uint32_t key_cut;  // key of the smallest kept logit
    uint64_t nk;       // kept tokens
    uint64_t zk;       // their fixed-point mass
    int32_t token;
};

// Row constants for a maximum zm (the global maximum, or a lower bound of it).
__device__ __forceinline__ RowCtx make_ctx(float zm, float T, float minp)
{
    RowCtx r;
    r.zmax = zm;
    r.T = T;
    r.invT = 1.f / T;
    if (!(r.invT <= FLT_MAX)) r.invT = FLT_MAX;
    r.minp = minp;
    r.L_lo = r.L_hi = 0.f;
    if (minp > 0.f) {
        const float L = -logf(minp);
        const float eps = 4e-6f * (1.f + L) + 1e-6f;
        r.L_lo = L - eps;
        r.L_hi = L + eps;
    }
    return r;
}

// zc: every token with z <= zc surely fails min-p (d(zc) > L_hi and d is monotone in z).  -inf when
// min-p is off or no such value was found.
__device__ __forceinline__ float minp_threshold(const RowCtx& r)
{
    if (!(r.minp > 0.f)) return -INFINITY;
    float c = r.zmax - r.L_hi * r.T;
    float step = fmaxf(fabsf(c) * 1e-6f, 1e-30f);
    int it = 0;
    while (!(dist(r, c) > r.L_hi) && it < 64) {
        c -= step;
        step *= 2.f;
        ++it;
    }
    return (dist(r, c) > r.L_hi) ? c : -INFINITY;
}

// Resolve a row whose min-p survivors are u.cd.sbuf[0, n) (n <= kCand, any order): top-k, top-p,
// race.  n <= 32 runs in warp 0 alone; larger n sorts with the whole CTA.
__device__ __forceinline__ RowResult resolve_candidates(Shared& s, const RowCtx& r, const RaceCtx& rc, uint32_t n,
                                                        bool topk_on, int32_t K, float P)
{
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    RowResult out;
    if (n <= 32) {
        if (tid < 32) {
            const WarpResult wr = warp_resolve(s.u.cd.sbuf, r, rc, n, topk_on, K, P);
            if (lane == 0) {
                s.bu[4] = wr.key_cut;
                s.bu[5] = wr.nk;
                s.b64[0] = wr.zk;
                s.bu[6] = (uint32_t)wr.token;
            }
        }
        cta_sync();
        out.key_cut = s.bu[4];
        out.nk = s.bu[5];
        out.zk = s.b64[0];
        out.token = (int32_t)s.bu[6];
        cta_sync();
        return out;
    }
    block_sort_desc(s, (int)n);
    prefix_masses(s, r, (int)n);
    int nS = (int)n;
    uint64_t ZS = s.u.cd.pre[n];
    if (topk_on && n > (uint32_t)K) {
        Crit ck;
        ck.by_mass = false;
        ck.tcnt = (uint64_t)K;
        ck.tmass = 0.0;
        const Sel sk = walk_classes(s, (int)n, ck, 0, 0);
        nS = (int)sk.cnt;
        ZS = sk.mass;
    }
    out.nk = (uint64_t)nS;
    out.zk = ZS;
    if (P < 1.f) {
        Crit cp;
        cp.by_mass = P > 0.f;
        cp.tcnt = 1;
        cp.tmass = (double)P * (double)ZS;
        const Sel sp = walk_classes(s, nS, cp, 0, 0);
        out.nk = sp.cnt;
        out.zk = sp.mass;
    }
    out.key_cut = sb_key(s.u.cd.sbuf[out.nk - 1]);
    // race over the kept prefix (one entry per thread: n <= kCand == kThreads)
    float k32 = -INFINITY, u = 0.f, z = 0.f;
    int32_t idx = 0x7FFFFFFF;
    if (tid < (int)out.nk) {
        const uint64_t v = s.u.cd.sbuf[tid];
        z = key_to_float(sb_key(v));
        idx = sb_idx(v);
        u = race_u(rc, idx);
        k32 = race_key32(dist(r, z), u);
    }
    float m32 = k32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m32 = fmaxf(m32, __shfl_xor_sync(0xFFFFFFFFu, m32, o));
    cta_sync();
    if (lane == 0) s.rf[tid >> 5] = m32;
    cta_sync();
    m32 = s.rf[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m32 = fmaxf(m32, s.rf[w]);
    const float tol = race_tol(dist(r, key_to_float(out.key_cut)));
    const bool fin = tid < (int)out.nk && k32 >= m32 - tol;
    const int nfin = cta_sync_count(fin);
    if (nfin == 1) {
        if (fin) s.bu[6] = (uint32_t)idx;
        cta_sync();
        out.token = (int32_t)s.bu[6];
    } else {
        ArgBest mine;
        mine.key = -INFINITY;
        mine.idx = 0x7FFFFFFF;
        if (fin) {
            mine.key = race_key64(r, z, u);
            mine.idx = idx;
        }
        out.token = block_argbest(mine, s).idx;
    }
    cta_sync();
    return out;
}

// Renormalised probabilities of the kept set over every element a source covers.
template <typename Src>
__device__ __forceinline__ void write_probs(const Src& src, const Shared& s, const RowCtx& r, uint32_t key_cut,
                                            uint64_t zk, float* prow)
{
    const double z64 = (double)zk;
    src.for_each(s, [&](float z, int32_t i) {
        float pv = 0.f;
        if (z > -INFINITY && fkey(z) >= key_cut) pv = (float)((double)qmass_d(dist(r, z)) / z64);
        prow[i] = pv;
    });
}

// The general path: min-p survivors counted against the global maximum (threshold zc), then the
// top-k and top-p cuts -- from a sorted candidate list when there are few survivors, else located by
// a histogram over d and refined exactly -- then the race over the kept tokens of the source, with
// the optional probability row written in the same pass.  Starts with a topology barrier, so the
// caller's published values may still be read by other CTAs when it is entered.
template <typename Topo, typename Src>
__device__ RowResult general_path(Topo& topo, Shared& s, const Src& src, const RowCtx& r, float zc, bool topk_on,
                                  int32_t K, float P, const RaceCtx& rc, float* prow)
{
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    const uint32_t C = topo.C;
    topo.sync();  // nobody still reads the caller's lists or published values
    if (tid == 0) s.ncand = 0;
    cta_sync();
    uint32_t my_minkey = 0xFFFFFFFFu;
    uint32_t my_surv = 0;
    src.for_each(s, [&](float z, int32_t i) {
        if (!(z > zc)) return;
        if (!minp_ok(r, z, dist(r, z))) return;
        const uint32_t key = fkey(z);
        my_minkey = min(my_minkey, key);
        ++my_surv;
        if (*(volatile uint32_t*)&s.ncand < (uint32_t)kCand) {
            const uint32_t slot = atomicAdd(&s.ncand, 1u);
            if (slot < (uint32_t)kCand) {
                s.ckey[slot] = key;
                s.cidx[slot] = (uint32_t)i;
            }
        }
    });
    my_surv = warp_sum_u32(my_surv);
    my_minkey = warp_min_u32(my_minkey);
    if (lane == 0) {
        s.ra[tid >> 5] = my_surv;
        s.rb[tid >> 5] = my_minkey;
    }
    cta_sync();
    if (tid == 0) {
        uint32_t ns = 0, mk = 0xFFFFFFFFu;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            ns += s.ra[w];
            mk = min(mk, s.rb[w]);
        }
        s.pub_nsurv = ns;
        s.pub_gcnt = min(ns, (uint32_t)kCand);
        s.pub_minkey = mk;
    }
    topo.sync();
    if (tid < 32) {
        uint32_t ns = 0, mk = 0xFFFFFFFFu;
        if (lane < C) {
            ns = *topo.map(&s.pub_nsurv, lane);
            mk = *topo.map(&s.pub_minkey, lane);
        }
        ns = warp_sum_u32(ns);
        mk = warp_min_u32(mk);
        if (lane == 0) {
            s.bu[2] = ns;
            s.bu[3] = mk;
        }
    }
    cta_sync();
    const uint64_t NS0 = s.bu[2];
    RowResult res;
    res.key_cut = s.bu[3];
    res.nk = NS0;
    res.zk = 0;

    if (NS0 <= (uint64_t)kCand) {
        // ---- few survivors: sort them (in every CTA)
        const int n = gather_and_sort(topo, s);
        prefix_masses(s, r, n);
        int nS = n;
        uint64_t ZS = s.u.cd.pre[n];
        if (topk_on && (uint64_t)n > (uint64_t)K) {
            Crit ck;
            ck.by_mass = false;
            ck.tcnt = (uint64_t)K;
            ck.tmass = 0.0;
            const Sel sk = walk_classes(s, n, ck, 0, 0);
            nS = (int)sk.cnt;
            ZS = sk.mass;
        }
        res.nk = (uint64_t)nS;
        res.zk = ZS;
        if (P < 1.f) {
            Crit cp;
            cp.by_mass = P > 0.f;
            cp.tcnt = 1;
            cp.tmass = (double)P * (double)ZS;
            const Sel sp = walk_classes(s, nS, cp, 0, 0);
            res.nk = sp.cnt;
            res.zk = sp.mass;
        }
        res.key_cut = sb_key(s.u.cd.sbuf[res.nk - 1]);
    } else {
        // ---- many survivors: histogram-located cuts, refined exactly
        for (int b = tid; b < kBins; b += kThreads) {
            s.hcnt[b] = 0;
            s.hmass[b] = 0;
        }
        cta_sync();
        auto build_hist = [&](uint32_t key_floor) {
            src.for_each(s, [&](float z, int32_t) {
                if (!(z > zc)) return;
                if (fkey(z) < key_floor) return;
                const float d = dist(r, z);
                if (!minp_ok(r, z, d)) return;
                const int b = bin_of(d);
                atomicAdd(&s.hcnt[b], 1u);
                atomicAdd((unsigned long long*)&s.hmass[b], (unsigned long long)qmass_d(d));
            });
        };
        build_hist(0u);
        cluster_reduce_hist(topo, s, kBins);
        uint64_t ZS;
        {
            uint64_t tot;
            (void)block_exscan_u64(s.hmass[tid], s, &tot);  // kBins == kThreads
            ZS = tot;
        }
        uint64_t NS = NS0;
        if (topk_on && NS0 > (uint64_t)K) {
            Crit ck;
            ck.by_mass = false;
            ck.tcnt = (uint64_t)K;
            ck.tmass = 0.0;
            int bk;
            uint64_t c_at, a_at;
            scan_bins(s, kBins, ck, 0, 0, &bk, &c_at, &a_at);
            if (bk < 0) bk = 0;
            const Sel sk = refine_bin(topo, s, src, r, zc, bk, 0u, ck, c_at, a_at);
            res.key_cut = max(res.key_cut, sk.key);
            NS = sk.cnt;
            ZS = sk.mass;
            if (P < 1.f) {  // rebuild the histogram over S = {key >= key_cut} for the top-p scan
                topo.sync();
                for (int b = tid; b < kBins; b += kThreads) {
                    s.hcnt[b] = 0;
                    s.hmass[b] = 0;
                }
                cta_sync();
                build_hist(res.key_cut);
                cluster_reduce_hist(topo, s, kBins);
            }
        }
        res.nk = NS;
        res.zk = ZS;
        if (P < 1.f) {
            Crit cp;
            cp.by_mass = P > 0.f;
            cp.tcnt = 1;
            cp.tmass = (double)P * (double)ZS;
            int bp;
            uint64_t c_at, a_at;
            scan_bins(s, kBins, cp, 0, 0, &bp, &c_at, &a_at);
            if (bp < 0) bp = 0;
            const Sel sp = refine_bin(topo, s, src, r, zc, bp, res.key_cut, cp, c_at, a_at);
            res.key_cut = max(res.key_cut, sp.key);
            res.nk = sp.cnt;
            res.zk = sp.mass;
        }
    }

    // ---- race over the kept tokens of the source (+ probabilities): float keys first; the best
    //      two decide whether double precision is needed at all
    const float tol = race_tol(dist(r, key_to_float(res.key_cut)));
    const uint32_t kc = res.key_cut;
    const double zk = (double)res.zk;
    Top2 t2;
    t2.init();
    src.for_each(s, [&](float z, int32_t i) {
        const bool kept = (z > -INFINITY) && fkey(z) >= kc;
        if (prow) prow[i] = kept ? (float)((double)qmass_d(dist(r, z)) / zk) : 0.f;
        if (!kept) return;
        t2.add(race_key32(dist(r, z), race_u(rc, i)), i);
    });
    t2 = warp_top2(t2);
    cta_sync();
    if (lane == 0) {
        s.rab[tid >> 5].key = (double)t2.k1;
        s.rab[tid >> 5].idx = t2.i1;
        s.rf[tid >> 5] = t2.k2;
    }
    cta_sync();
    if (tid == 0) {
        Top2 b;
        b.init();
        for (int w = 0; w < kWarps; ++w) {
            Top2 x;
            x.k1 = (float)s.rab[w].key;
            x.i1 = s.rab[w].idx;
            x.k2 = s.rf[w];
            b.merge(x);
        }
        s.pub_k64 = (double)b.k1;  // published: best float key, its index, second float key
        s.pub_idx = b.i1;
        s.pub_max = b.k2;
    }
    topo.sync();
    if (tid < 32) {
        Top2 x;
        x.init();
        if (lane < C) {
            x.k1 = (float)*topo.map(&s.pub_k64, lane);
            x.i1 = *topo.map(&s.pub_idx, lane);
            x.k2 = *topo.map(&s.pub_max, lane);
        }
        x = warp_top2(x);
        if (lane == 0) {
            s.bf[1] = x.k1;
            s.bf[0] = x.k2;
            s.bu[6] = (uint32_t)x.i1;
        }
    }
    cta_sync();
    const float M1 = s.bf[1], M2 = s.bf[0];
    res.token = (int32_t)s.bu[6];
    if (!(M1 - M2 > tol)) {
        // near-tie: every kept token within tol of the best is re-evaluated in double precision
        ArgBest mine;
        mine.key = -INFINITY;
        mine.idx = 0x7FFFFFFF;
        src.for_each(s, [&](float z, int32_t i) {
            if (!((z > -INFINITY) && fkey(z) >= kc)) return;
            const float u = race_u(rc, i);
            if (race_key32(dist(r, z), u) >= M1 - tol) {
                const double k64 = race_key64(r, z, u);
                if (better(k64, i, mine.key, mine.idx)) {
                    mine.key = k64;
                    mine.idx = i;
                }
            }
        });
        mine = block_argbest(mine, s);
        topo.sync();  // everyone has read the published float keys
        if (tid == 0) {
            s.pub_k64 = mine.key;
            s.pub_idx = mine.idx;
        }
        topo.sync();
        if (tid < 32) {
            ArgBest x;
            x.key = -INFINITY;
            x.idx = 0x7FFFFFFF;
            if (lane < C) {
                x.key = *topo.map(&s.pub_k64, lane);
                x.idx = *topo.map(&s.pub_idx, lane);
            }
            x = warp_argbest(x);
            if (lane == 0) s.bu[6] = (uint32_t)x.idx;
        }
        cta_sync();
        res.token = (int32_t)s.bu[6];
    }
    cta_sync();
    return res;
}

// Per-row outputs (thread 0 of the writing CTA).
__device__ __forceinline__ void write_row(const Args& a, int64_t row, int32_t token, int32_t status, float cutoff,
                                          int32_t kept)
{
    a.out_token[row] = token;
    if (a.out_status) a.out_status[row] = status;
    if (a.out_cutoff) a.out_cutoff[row] = cutoff;
    if (a.out_kept) a.out_kept[row] = kept;
}

}  // namespace tps
