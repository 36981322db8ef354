// tps_kernel.cuh -- the row sampler: one thread-block cluster per row, the row held in the
// cluster's shared memory.
//
// Each of the C CTAs of a cluster bulk-copies one contiguous 16-byte-aligned slice of the row from
// HBM into its own shared memory (one read of the row, no multicast); the ragged head and tail of
// an unaligned row are fetched with plain loads.  Everything after that reads shared memory only,
// and the CTAs exchange small reductions through distributed shared memory:
//
//   A  zmax (NaN-propagating max) -> row status, greedy branch;
//   B  one pass: d = (zmax - z)/T, min-p survival, 512-bin histogram over d of {count, exact
//      fixed-point mass}, and the survivors appended to a candidate list;
//   C  few survivors (<= 1024): every CTA gathers all candidates, sorts them by (logit desc,
//      index asc) and walks the classes of equal logits: top-k cut by count, top-p cut by mass,
//      then the exponential race over the kept prefix;
//      many survivors: the histogram locates the bin holding each cut; the cut's class is then
//      resolved exactly by gathering that bin's tokens (or by further sub-histograms over the
//      logit's order-preserving key until few enough remain or a single value is left);
//   D  the race over the kept tokens (those with logit >= the cut), and the optional output row
//      of renormalised probabilities.
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
constexpr int kBins = 512;            // level-1 bins over d, width 1/16 (last bin: d >= 31.9375)
constexpr float kBinScale = 16.f;
constexpr int kSubBins = 512;         // sub-bins over a key interval
constexpr int kCand = 1024;           // candidates resolved by sorting, per CTA and per cluster
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
    // --- values other CTAs of the cluster read through distributed shared memory
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
    uint32_t ru[kWarps];
    uint32_t ru2[kWarps];
    uint64_t r64[kWarps];
    ArgBest rab[kWarps];
    uint32_t bu[4];
    uint64_t b64[2];
    // --- histograms: local, then (after the cluster reduction) the full reduced histogram
    uint32_t hcnt[kBins];
    uint64_t hmass[kBins];
    // --- this CTA's share of the reduced histogram (read by the other CTAs)
    uint32_t rcnt[kBins];
    uint64_t rmass[kBins];
    // --- candidates
    uint32_t ncand;
    uint32_t ckey[kCand];
    uint32_t cidx[kCand];
    uint64_t sbuf[kCand];     // gathered (key << 32 | ~index), sorted descending
    uint64_t pre[kCand + 1];  // exclusive prefix of the fixed-point masses along sbuf
};

// ---------------------------------------------------------------------------------------------
// Block-level helpers (every thread of the CTA must call them).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float block_max_nan(float v, Shared& s)
{
    v = warp_max_nan(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s.rf[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = s.rf[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = fmax_nan(r, s.rf[w]);
    return r;
}

__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, Shared& s)
{
    v = warp_min_u32(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = s.ru[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = min(r, s.ru[w]);
    return r;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, Shared& s)
{
    v = warp_max_u32(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s.ru2[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = s.ru2[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = max(r, s.ru2[w]);
    return r;
}

__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, Shared& s)
{
    v = warp_sum_u32(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s.ru[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) r += s.ru[w];
    return r;
}

__device__ __forceinline__ ArgBest block_argbest(ArgBest a, Shared& s)
{
    a = warp_argbest(a);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s.rab[threadIdx.x >> 5] = a;
    __syncthreads();
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
    __syncthreads();
    if (lane == 31) s.r64[warp] = x;
    __syncthreads();
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
// The slice of the row this CTA holds.
// ---------------------------------------------------------------------------------------------
template <typename TIn>
struct Slice {
    const uint4* vec;  // shared-memory vectors of Elem<TIn>::kPerVec elements
    int nvec;
    int64_t elem0;     // row index of the first element of vec[0]

    // Apply f(z, i) to every element of the slice (vectors, then the ragged extras).
    template <typename F>
    __device__ __forceinline__ void for_each(const Shared& s, F&& f) const
    {
        using E = Elem<TIn>;
        for (int v = threadIdx.x; v < nvec; v += kThreads) {
            float z[E::kPerVec];
            E::unpack(vec[v], z);
            const int32_t i0 = (int32_t)(elem0 + (int64_t)v * E::kPerVec);
#pragma unroll
            for (int j = 0; j < E::kPerVec; ++j) f(z[j], i0 + j);
        }
        for (int x = threadIdx.x; x < s.nx; x += kThreads) f(s.xz[x], s.xi[x]);
    }
};

__device__ __forceinline__ int bin_of(float d)
{
    return min(__float2int_rz(d * kBinScale), kBins - 1);
}

// Cluster-wide sum of the local histogram hcnt/hmass[0, nb) into hcnt/hmass of every CTA.
// Step 1: CTA c sums its share of bins over all CTAs into rcnt/rmass; step 2: every CTA copies
// all shares back into its own hcnt/hmass.
__device__ __forceinline__ void cluster_reduce_hist(cg::cluster_group& cluster, Shared& s, int nb,
                                                    uint32_t C, uint32_t rank)
{
    cluster.sync();  // all local histograms complete
    const int per = (nb + (int)C - 1) / (int)C;
    const int b0 = (int)rank * per, b1 = min(nb, b0 + per);
    for (int b = b0 + (int)threadIdx.x; b < b1; b += kThreads) {
        uint32_t c = 0;
        uint64_t m = 0;
        for (uint32_t r = 0; r < C; ++r) {
            c += *cluster.map_shared_rank(&s.hcnt[b], r);
            m += *cluster.map_shared_rank(&s.hmass[b], r);
        }
        s.rcnt[b] = c;
        s.rmass[b] = m;
    }
    cluster.sync();  // all shares complete; nobody reads hcnt/hmass of another CTA any more
    for (int b = threadIdx.x; b < nb; b += kThreads) {
        const uint32_t owner = (uint32_t)(b / per);
        s.hcnt[b] = *cluster.map_shared_rank(&s.rcnt[b], owner);
        s.hmass[b] = *cluster.map_shared_rank(&s.rmass[b], owner);
    }
    __syncthreads();
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
// last non-empty bin whose (count, mass) above satisfies the criterion.  Bins after `cap` are
// ignored and bin `cap` counts as (cap_cnt, cap_mass).
__device__ __forceinline__ void scan_bins(Shared& s, int nb, const Crit& cr, int cap, uint32_t cap_cnt,
                                          uint64_t cap_mass, uint64_t C0, uint64_t A0, int* out_bin,
                                          uint64_t* out_c, uint64_t* out_a)
{
    // nb <= 2 * kThreads: each thread owns bins 2t and 2t + 1.
    const int b0 = 2 * threadIdx.x, b1 = b0 + 1;
    auto eff_c = [&](int b) -> uint64_t {
        if (b >= nb || b > cap) return 0;
        return b == cap ? cap_cnt : s.hcnt[b];
    };
    auto eff_m = [&](int b) -> uint64_t {
        if (b >= nb || b > cap) return 0;
        return b == cap ? cap_mass : s.hmass[b];
    };
    const uint64_t c0 = eff_c(b0), c1 = eff_c(b1), m0 = eff_m(b0), m1 = eff_m(b1);
    uint64_t tot;
    const uint64_t cpre = block_exscan_u64(c0 + c1, s, &tot);
    const uint64_t mpre = block_exscan_u64(m0 + m1, s, &tot);
    uint32_t best = 0;  // bin + 1, 0 = none
    if (c0 > 0 && cr.keep(C0 + cpre, A0 + mpre)) best = b0 + 1;
    if (c1 > 0 && cr.keep(C0 + cpre + c0, A0 + mpre + m0)) best = b1 + 1;
    const uint32_t bb = block_max_u32(best, s);
    // Publish the prefix of the chosen bin.
    if (bb != 0) {
        const int b = (int)bb - 1;
        if (b == b0) {
            s.b64[0] = C0 + cpre;
            s.b64[1] = A0 + mpre;
        } else if (b == b1) {
            s.b64[0] = C0 + cpre + c0;
            s.b64[1] = A0 + mpre + m0;
        }
    }
    __syncthreads();
    *out_bin = (int)bb - 1;
    *out_c = bb ? s.b64[0] : C0;
    *out_a = bb ? s.b64[1] : A0;
    __syncthreads();
}

// Sort sbuf[0, n) descending (bitonic, padded with zeros to a power of two).
__device__ __forceinline__ void block_sort_desc(Shared& s, int n)
{
    int np = 2;
    while (np < n) np <<= 1;
    for (int i = n + (int)threadIdx.x; i < np; i += kThreads) s.sbuf[i] = 0;
    __syncthreads();
    for (int k2 = 2; k2 <= np; k2 <<= 1) {
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < (np >> 1); i += kThreads) {
                const int lo = 2 * j * (i / j) + (i % j), hi = lo + j;
                const bool desc = (lo & k2) == 0;
                const uint64_t x = s.sbuf[lo], y = s.sbuf[hi];
                if (desc ? (x < y) : (x > y)) {
                    s.sbuf[lo] = y;
                    s.sbuf[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

__device__ __forceinline__ uint32_t sb_key(uint64_t v) { return (uint32_t)(v >> 32); }
__device__ __forceinline__ int32_t sb_idx(uint64_t v) { return (int32_t)(~(uint32_t)v); }

// Fill pre[0, n] with the exclusive prefix of the fixed-point masses of sbuf[0, n).
__device__ __forceinline__ void prefix_masses(Shared& s, const RowCtx& r, int n)
{
    // up to kCand = 4 * kThreads entries: each thread takes 4 consecutive ones
    uint64_t q[4];
    uint64_t local = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int t = 4 * threadIdx.x + j;
        q[j] = (t < n) ? qmass_d(dist(r, key_to_float(sb_key(s.sbuf[t])))) : 0;
        local += q[j];
    }
    uint64_t tot;
    uint64_t run = block_exscan_u64(local, s, &tot);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int t = 4 * threadIdx.x + j;
        if (t < n) s.pre[t] = run;
        run += q[j];
    }
    if (threadIdx.x == 0) s.pre[n] = tot;
    __syncthreads();
}

// Walk the classes of the sorted candidates sbuf[0, n) (n <= the list length) and return the
// last class whose (count, mass) above -- offset by (C0, A0) -- satisfies the criterion.
__device__ __forceinline__ Sel walk_classes(Shared& s, int n, const Crit& cr, uint64_t C0, uint64_t A0)
{
    uint32_t best = 0;  // position + 1 of the chosen class start
    for (int t = threadIdx.x; t < n; t += kThreads) {
        const uint32_t kt = sb_key(s.sbuf[t]);
        const bool start = (t == 0) || sb_key(s.sbuf[t - 1]) != kt;
        if (start && cr.keep(C0 + (uint64_t)t, A0 + s.pre[t])) best = max(best, (uint32_t)t + 1u);
    }
    const uint32_t sb = block_max_u32(best, s);
    const int st = sb ? (int)sb - 1 : 0;
    uint32_t end = (uint32_t)n;
    for (int t = st + 1 + (int)threadIdx.x; t < n; t += kThreads)
        if (sb_key(s.sbuf[t]) != sb_key(s.sbuf[t - 1])) end = min(end, (uint32_t)t);
    const uint32_t e = block_min_u32(end, s);
    Sel out;
    out.key = sb_key(s.sbuf[st]);
    out.cnt = C0 + e;
    out.mass = A0 + s.pre[e];
    __syncthreads();
    return out;
}

// Copy every CTA's candidate list (counts published in pub_gcnt) into sbuf, sort it.
__device__ __forceinline__ int gather_and_sort(cg::cluster_group& cluster, Shared& s, uint32_t C)
{
    uint32_t off = 0;
    for (uint32_t rr = 0; rr < C; ++rr) {
        const uint32_t n = *cluster.map_shared_rank(&s.pub_gcnt, rr);
        const uint32_t* rk = cluster.map_shared_rank(&s.ckey[0], rr);
        const uint32_t* ri = cluster.map_shared_rank(&s.cidx[0], rr);
        for (uint32_t t = threadIdx.x; t < n; t += kThreads)
            s.sbuf[off + t] = ((uint64_t)rk[t] << 32) | (uint64_t)(~ri[t]);
        off += n;
    }
    __syncthreads();
    block_sort_desc(s, (int)off);
    return (int)off;
}

// Race key in float (for pruning) and in double (for the decision) of kept token i.
struct RaceCtx {
    uint32_t k0, k1;    // Philox key = seed
    uint32_t row, s_lo, s_hi;
    float dmax_tol;     // pruning margin
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

// Refine the cut inside level-1 bin `bin` (tokens with key >= key_lo that survive min-p), given
// the (count, mass) of the survivors above the bin.  Exact: ends with a sorted candidate list or
// with a single logit value.
template <typename TIn>
__device__ Sel refine_bin(cg::cluster_group& cluster, Shared& s, const Slice<TIn>& sl, const RowCtx& r,
                          uint32_t C, int bin, uint32_t key_lo, const Crit& cr, uint64_t C0, uint64_t A0)
{
    // Phase 1: gather the bin (and its key range).
    uint32_t klo = 0, khi = 0xFFFFFFFFu;
    bool by_bin = true;
    for (int iter = 0; iter < 8; ++iter) {
        cluster.sync();  // nobody still reads my candidate list or published counts
        if (threadIdx.x == 0) s.ncand = 0;
        __syncthreads();
        uint32_t lcnt = 0, lmin = 0xFFFFFFFFu, lmax = 0;
        sl.for_each(s, [&](float z, int32_t i) {
            if (!(z > -INFINITY)) return;
            const uint32_t key = fkey(z);
            if (key < key_lo || key < klo || key > khi) return;
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
            s.pub_gcnt = cnt;
            s.pub_gkmin = kmn;
            s.pub_gkmax = kmx;
        }
        cluster.sync();
        uint64_t total = 0;
        uint32_t gmin = 0xFFFFFFFFu, gmax = 0;
        for (uint32_t rr = 0; rr < C; ++rr) {
            total += *cluster.map_shared_rank(&s.pub_gcnt, rr);
            gmin = min(gmin, *cluster.map_shared_rank(&s.pub_gkmin, rr));
            gmax = max(gmax, *cluster.map_shared_rank(&s.pub_gkmax, rr));
        }
        if (total == 0) {  // cannot happen for a bin chosen as non-empty; keep the bound
            Sel z0;
            z0.key = key_lo;
            z0.cnt = C0;
            z0.mass = A0;
            return z0;
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
            const int n = gather_and_sort(cluster, s, C);
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
        __syncthreads();
        const uint32_t lo = klo, hi = khi;
        sl.for_each(s, [&](float z, int32_t) {
            if (!(z > -INFINITY)) return;
            const uint32_t key = fkey(z);
            if (key < key_lo || key < lo || key > hi) return;
            const float d = dist(r, z);
            if (!minp_ok(r, z, d)) return;
            const int sb = (int)((hi - key) >> sh);
            atomicAdd(&s.hcnt[sb], 1u);
            atomicAdd((unsigned long long*)&s.hmass[sb], (unsigned long long)qmass_d(d));
        });
        cluster_reduce_hist(cluster, s, kSubBins, C, cluster.block_rank());
        int jb;
        uint64_t c_at, a_at;
        scan_bins(s, nsub, cr, nsub - 1, s.hcnt[nsub - 1], s.hmass[nsub - 1], C0, A0, &jb, &c_at, &a_at);
        if (jb < 0) jb = 0;
        C0 = c_at;
        A0 = a_at;
        const uint64_t top = (uint64_t)hi - ((uint64_t)jb << sh);
        const uint64_t width = (uint64_t)1 << sh;
        const uint64_t bot = (top + 1 >= width) ? top + 1 - width : 0;
        khi = (uint32_t)top;
        klo = (uint32_t)max((uint64_t)lo, bot);
    }
    // Unreachable in practice (each split shrinks the 32-bit range by 2^9); keep a valid answer.
    Sel o;
    o.key = khi;
    o.cnt = C0;
    o.mass = A0;
    return o;
}

// ---------------------------------------------------------------------------------------------
// The kernel.  Grid: B * C CTAs in clusters of C along x; cluster q samples row q.
// ---------------------------------------------------------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1) sample_rows_kernel(const Args a)
{
    using E = Elem<TIn>;
    constexpr int EPV = E::kPerVec;
    constexpr int ES = E::kBytes;
    extern __shared__ __align__(128) unsigned char dsmem[];

    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t C = cluster.num_blocks();
    const uint32_t rank = cluster.block_rank();
    const int64_t row = (int64_t)(blockIdx.x / C);
    Shared& s = *reinterpret_cast<Shared*>(dsmem + a.slice_cap);
    const int tid = threadIdx.x;

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

    // ---- stage the slice: one bulk copy (split in 32 KB pieces) completing on an mbarrier
    const int my_head = (rank == 0) ? (int)nhead : 0;
    const int my_tail = (rank == C - 1) ? (int)ntail : 0;
    if (tid == 0) {
        s.nx = my_head + my_tail;
        if (bytes > 0) mbar_init(&s.mbar, 1);
    }
    __syncthreads();
    if (tid == 0 && bytes > 0) {
        mbar_arrive_expect_tx(&s.mbar, bytes);
        const unsigned char* src = reinterpret_cast<const unsigned char*>(a0) + v_lo * 16;
        for (uint32_t off = 0; off < bytes; off += 32768u)
            bulk_g2s(dsmem + off, src + off, min(32768u, bytes - off), &s.mbar);
    }
    if (tid < my_head) {
        s.xz[tid] = E::load1(rowp, tid);
        s.xi[tid] = tid;
    } else if (tid < my_head + my_tail) {
        const int64_t i = a.V - ntail + (tid - my_head);
        s.xz[tid] = E::load1(rowp, i);
        s.xi[tid] = (int32_t)i;
    }
    uint32_t timed_out = 0;
    if (bytes > 0 && !mbar_wait_bounded(&s.mbar, 0, kWaitLimitNs)) timed_out = 1;
    __syncthreads();

    // ---- A: zmax with NaN propagation (a NaN anywhere makes the maximum NaN)
    float vmax = -INFINITY;
    if (!timed_out) sl.for_each(s, [&](float z, int32_t) { vmax = fmax_nan(vmax, z); });
    vmax = block_max_nan(vmax, s);
    const uint32_t any_to = block_max_u32(timed_out, s);
    if (tid == 0) {
        s.pub_max = vmax;
        s.pub_timeout = any_to;
    }
    cluster.sync();
    float zmax = -INFINITY;
    uint32_t cl_timeout = 0;
    for (uint32_t rr = 0; rr < C; ++rr) {
        zmax = fmax_nan(zmax, *cluster.map_shared_rank(&s.pub_max, rr));
        cl_timeout |= *cluster.map_shared_rank(&s.pub_timeout, rr);
    }

    const float T = a.temperature[row];
    const float P = a.top_p[row];
    const float MP = a.min_p[row];
    const int32_t K = a.top_k[row];
    const uint64_t seed = a.seed[row];

    int32_t status = kRowOk;
    if (cl_timeout) status = kRowTimeout;
    else if (isnan(zmax) || zmax == INFINITY) status = kRowNan;
    else if (!isfinite(T) || !isfinite(P) || !isfinite(MP)) status = kRowBadParam;
    else if (zmax == -INFINITY) status = kRowAllMasked;

    float* prow = a.out_probs ? a.out_probs + row * a.V : nullptr;
    const bool writer = (rank == 0) && (tid == 0);

    if (status != kRowOk) {
        if (prow && !timed_out) sl.for_each(s, [&](float, int32_t i) { prow[i] = 0.f; });
        if (prow && timed_out) {
            for (int64_t i = sl.elem0 + tid; i < sl.elem0 + (int64_t)nvec * EPV; i += kThreads) prow[i] = 0.f;
            for (int x = tid; x < s.nx; x += kThreads) prow[s.xi[x]] = 0.f;
        }
        if (writer) {
            a.out_token[row] = -1;
            if (a.out_status) a.out_status[row] = status;
            if (a.out_cutoff) a.out_cutoff[row] = __uint_as_float(0x7FC00000u);
            if (a.out_kept) a.out_kept[row] = 0;
        }
        // A copy still in flight after a timeout must land before the shared memory is released.
        if (timed_out && bytes > 0) (void)mbar_wait_bounded(&s.mbar, 0, kWaitLimitNs);
        cluster.sync();
        return;
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
        uint32_t arg = 0xFFFFFFFFu;
        for (uint32_t rr = 0; rr < C; ++rr) arg = min(arg, *cluster.map_shared_rank(&s.pub_minidx, rr));
        if (prow) sl.for_each(s, [&](float, int32_t i) { prow[i] = ((uint32_t)i == arg) ? 1.f : 0.f; });
        if (writer) {
            a.out_token[row] = (int32_t)arg;
            if (a.out_status) a.out_status[row] = kRowOk;
            if (a.out_cutoff) a.out_cutoff[row] = zmax;
            if (a.out_kept) a.out_kept[row] = 1;
        }
        cluster.sync();
        return;
    }

    // ---- row constants
    RowCtx r;
    r.zmax = zmax;
    r.T = T;
    r.invT = 1.f / T;
    if (!(r.invT <= FLT_MAX)) r.invT = FLT_MAX;
    r.minp = (MP > 0.f) ? fminf(MP, 1.f) : 0.f;
    r.L_lo = r.L_hi = 0.f;
    if (r.minp > 0.f) {
        const float L = -logf(r.minp);
        const float eps = 4e-6f * (1.f + L) + 1e-6f;
        r.L_lo = L - eps;
        r.L_hi = L + eps;
    }

    // ---- B: min-p survivors -> histogram over d + candidate list
    for (int b = tid; b < kBins; b += kThreads) {
        s.hcnt[b] = 0;
        s.hmass[b] = 0;
    }
    if (tid == 0) s.ncand = 0;
    __syncthreads();
    uint32_t my_minkey = 0xFFFFFFFFu;
    uint32_t my_surv = 0;
    sl.for_each(s, [&](float z, int32_t i) {
        if (!(z > -INFINITY)) return;
        const float d = dist(r, z);
        if (!minp_ok(r, z, d)) return;
        const uint32_t key = fkey(z);
        const int b = bin_of(d);
        atomicAdd(&s.hcnt[b], 1u);
        atomicAdd((unsigned long long*)&s.hmass[b], (unsigned long long)qmass_d(d));
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
    const uint32_t nsurv = block_sum_u32(my_surv, s);
    const uint32_t mink = block_min_u32(my_minkey, s);
    if (tid == 0) {
        s.pub_nsurv = nsurv;
        s.pub_gcnt = min(nsurv, (uint32_t)kCand);
        s.pub_minkey = mink;
    }
    cluster.sync();
    uint64_t NS0 = 0;
    uint32_t key_minp = 0xFFFFFFFFu;
    for (uint32_t rr = 0; rr < C; ++rr) {
        NS0 += *cluster.map_shared_rank(&s.pub_nsurv, rr);
        key_minp = min(key_minp, *cluster.map_shared_rank(&s.pub_minkey, rr));
    }

    const bool topk_on = (K > 0) && ((int64_t)K < a.V);
    uint32_t key_cut = key_minp;
    uint64_t NK = NS0, ZK = 0;

    RaceCtx rc;
    rc.k0 = (uint32_t)seed;
    rc.k1 = (uint32_t)(seed >> 32);
    rc.row = (uint32_t)row;
    rc.s_lo = (uint32_t)a.step;
    rc.s_hi = (uint32_t)(a.step >> 32);

    ArgBest win;
    win.key = -INFINITY;
    win.idx = 0x7FFFFFFF;

    if (NS0 <= (uint64_t)kCand) {
        // ---- C (few survivors): sort all candidates and walk their classes, in every CTA
        const int n = gather_and_sort(cluster, s, C);
        prefix_masses(s, r, n);
        int nS = n;
        uint64_t ZS = s.pre[n];
        if (topk_on && (uint64_t)n > (uint64_t)K) {
            Crit ck;
            ck.by_mass = false;
            ck.tcnt = (uint64_t)K;
            ck.tmass = 0.0;
            const Sel sk = walk_classes(s, n, ck, 0, 0);
            key_cut = max(key_cut, sk.key);
            nS = (int)sk.cnt;
            ZS = sk.mass;
        }
        NK = (uint64_t)nS;
        ZK = ZS;
        if (P < 1.f) {
            Crit cp;
            cp.by_mass = P > 0.f;
            cp.tcnt = 1;
            cp.tmass = (double)P * (double)ZS;
            const Sel sp = walk_classes(s, nS, cp, 0, 0);
            key_cut = max(key_cut, sp.key);
            NK = sp.cnt;
            ZK = sp.mass;
        }
        // Race over the kept prefix: float keys locate the finalists, double keys decide.
        const int nk = (int)NK;
        const float dcut = dist(r, key_to_float(key_cut));
        const float tol = 1e-5f + 1e-6f * dcut;
        float k32 = -INFINITY;
        // kept <= kCand = 4 * kThreads: a thread holds up to 4 entries; keep the best locally.
        float kk[4];
        float uu[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = tid + j * kThreads;
            kk[j] = -INFINITY;
            uu[j] = 0.f;
            if (t < nk) {
                const uint64_t v = s.sbuf[t];
                const float z = key_to_float(sb_key(v));
                uu[j] = race_u(rc, sb_idx(v));
                kk[j] = race_key32(dist(r, z), uu[j]);
                k32 = fmaxf(k32, kk[j]);
            }
        }
        // block max of the float keys
        float m32 = k32;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m32 = fmaxf(m32, __shfl_xor_sync(0xFFFFFFFFu, m32, o));
        __syncthreads();
        if ((tid & 31) == 0) s.rf[tid >> 5] = m32;
        __syncthreads();
        m32 = s.rf[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) m32 = fmaxf(m32, s.rf[w]);
        ArgBest mine;
        mine.key = -INFINITY;
        mine.idx = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = tid + j * kThreads;
            if (t < nk && kk[j] >= m32 - tol) {
                const uint64_t v = s.sbuf[t];
                const double k64 = race_key64(r, key_to_float(sb_key(v)), uu[j]);
                if (better(k64, sb_idx(v), mine.key, mine.idx)) {
                    mine.key = k64;
                    mine.idx = sb_idx(v);
                }
            }
        }
        win = block_argbest(mine, s);
        // optional probabilities over the slice
        if (prow) {
            const double zk = (double)ZK;
            const uint32_t kc = key_cut;
            sl.for_each(s, [&](float z, int32_t i) {
                float pv = 0.f;
                if (z > -INFINITY && fkey(z) >= kc) pv = (float)((double)qmass_d(dist(r, z)) / zk);
                prow[i] = pv;
            });
        }
    } else {
        // ---- C (many survivors): histogram-located cuts, refined exactly
        cluster_reduce_hist(cluster, s, kBins, C, rank);
        uint64_t Z0 = 0;
        {
            uint64_t m = 0;
            for (int b = tid; b < kBins; b += kThreads) m += s.hmass[b];
            uint64_t tot;
            (void)block_exscan_u64(m, s, &tot);
            Z0 = tot;
        }
        uint64_t NS = NS0, ZS = Z0;
        int cap = kBins - 1;
        uint32_t cap_cnt = s.hcnt[kBins - 1];
        uint64_t cap_mass = s.hmass[kBins - 1];
        if (topk_on && NS0 > (uint64_t)K) {
            Crit ck;
            ck.by_mass = false;
            ck.tcnt = (uint64_t)K;
            ck.tmass = 0.0;
            int bk;
            uint64_t c_at, a_at;
            scan_bins(s, kBins, ck, cap, cap_cnt, cap_mass, 0, 0, &bk, &c_at, &a_at);
            if (bk < 0) bk = 0;
            const Sel sk = refine_bin<TIn>(cluster, s, sl, r, C, bk, 0u, ck, c_at, a_at);
            key_cut = max(key_cut, sk.key);
            NS = sk.cnt;
            ZS = sk.mass;
            // The refinement may have reused the histogram; rebuild it over S for the top-p scan.
            if (P < 1.f) {
                cluster.sync();
                for (int b = tid; b < kBins; b += kThreads) {
                    s.hcnt[b] = 0;
                    s.hmass[b] = 0;
                }
                __syncthreads();
                const uint32_t kc = key_cut;
                sl.for_each(s, [&](float z, int32_t) {
                    if (!(z > -INFINITY)) return;
                    if (fkey(z) < kc) return;
                    const float d = dist(r, z);
                    if (!minp_ok(r, z, d)) return;
                    const int b = bin_of(d);
                    atomicAdd(&s.hcnt[b], 1u);
                    atomicAdd((unsigned long long*)&s.hmass[b], (unsigned long long)qmass_d(d));
                });
                cluster_reduce_hist(cluster, s, kBins, C, rank);
            }
            cap = kBins - 1;
            cap_cnt = s.hcnt[kBins - 1];
            cap_mass = s.hmass[kBins - 1];
        }
        NK = NS;
        ZK = ZS;
        if (P < 1.f) {
            Crit cp;
            cp.by_mass = P > 0.f;
            cp.tcnt = 1;
            cp.tmass = (double)P * (double)ZS;
            int bp;
            uint64_t c_at, a_at;
            scan_bins(s, kBins, cp, cap, cap_cnt, cap_mass, 0, 0, &bp, &c_at, &a_at);
            if (bp < 0) bp = 0;
            const Sel sp = refine_bin<TIn>(cluster, s, sl, r, C, bp, key_cut, cp, c_at, a_at);
            key_cut = max(key_cut, sp.key);
            NK = sp.cnt;
            ZK = sp.mass;
        }
        // ---- D: race over the kept tokens of the slice (+ probabilities)
        const float dcut = dist(r, key_to_float(key_cut));
        const float tol = 1e-5f + 1e-6f * dcut;
        const uint32_t kc = key_cut;
        const double zk = (double)ZK;
        float best32 = -INFINITY;
        ArgBest mine;
        mine.key = -INFINITY;
        mine.idx = 0x7FFFFFFF;
        sl.for_each(s, [&](float z, int32_t i) {
            const bool kept = (z > -INFINITY) && fkey(z) >= kc;
            if (prow) prow[i] = kept ? (float)((double)qmass_d(dist(r, z)) / zk) : 0.f;
            if (!kept) return;
            const float u = race_u(rc, i);
            const float k32 = race_key32(dist(r, z), u);
            if (k32 >= best32 - tol) {
                const double k64 = race_key64(r, z, u);
                if (better(k64, i, mine.key, mine.idx)) {
                    mine.key = k64;
                    mine.idx = i;
                }
            }
            best32 = fmaxf(best32, k32);
        });
        mine = block_argbest(mine, s);
        if (tid == 0) {
            s.pub_k64 = mine.key;
            s.pub_idx = mine.idx;
        }
        cluster.sync();
        for (uint32_t rr = 0; rr < C; ++rr) {
            const double kq = *cluster.map_shared_rank(&s.pub_k64, rr);
            const int32_t iq = *cluster.map_shared_rank(&s.pub_idx, rr);
            if (better(kq, iq, win.key, win.idx)) {
                win.key = kq;
                win.idx = iq;
            }
        }
    }

    if (writer) {
        a.out_token[row] = win.idx;
        if (a.out_status) a.out_status[row] = kRowOk;
        if (a.out_cutoff) a.out_cutoff[row] = key_to_float(key_cut);
        if (a.out_kept) a.out_kept[row] = (int32_t)NK;
    }
    cluster.sync();  // keep this CTA's shared memory alive until every remote read is done
}

}  // namespace tps
