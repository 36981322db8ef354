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
constexpr int kFineBins = 512;        // count bins over d, width 1/16 (last bin: d >= 511/16)
constexpr float kFineScale = 16.f;
constexpr int kRaceQueue = 96;        // per-warp queue of vectors with tokens to race
constexpr int kSubBins = 128;         // sub-bins over a key interval (exact refinement)
constexpr int kMaxWin = 32;           // groups of fine bins in a top-p window
constexpr int kMaxTop = 32;           // top tokens a call may report per row
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
    float* out_logprob;  // ln P(token) under the renormalised kept distribution, or null
    int32_t n_top;           // top tokens reported per row (0 .. kMaxTop)
    int32_t* out_top_idx;    // [B, n_top]: the most probable kept tokens, or null
    float* out_top_logprob;  // [B, n_top]: their ln P
    uint32_t slice_cap;  // bytes reserved for the slice at the start of dynamic shared memory
    uint32_t route;      // which rows the kernel samples (RowRoute)
    // Streaming kernel's work: rows [0, b_whole) are claimed whole; each of the last nsplit rows is
    // claimed as nseg segments, merged by the CTA that finishes a row's last segment.
    void* scratch;       // global scratch of the call (ScratchLayout), cleared before the kernel claims
    int64_t b_whole;
    int64_t nsplit;
    int32_t nseg;
    uint64_t wait_ns;     // limit of the consumers' waits in the streaming kernel (kWaitLimitNs; shorter in a test)
    int64_t stall_chunk;  // test hook: chunk whose copy CTA 0 of the streaming kernel withholds (-1: none)
};

// Which rows a kernel samples.  A large batch is split between the two kernels: the streaming
// kernel takes every row but those routed_to_cluster() selects and lists those in the scratch; the
// cluster kernel, launched behind it, takes the listed rows.
enum RowRoute : uint32_t { kRouteAll = 0, kRouteStream = 1, kRouteList = 2 };

// ---------------------------------------------------------------------------------------------
// Global scratch of one streaming call.  Work is claimed dynamically: a claim q < b_whole is row q,
// whole; a claim q >= b_whole is segment (q - b_whole) % nseg of row b_whole + (q - b_whole) / nseg.
// A CTA's first claim is its block index; later claims come from `claim`.  Each segment of a split
// row publishes a partial result (its maximum and the tokens it listed); the CTA whose arrival on
// the row's counter completes the count merges them.  Everything that must start at zero (the
// header and the arrival counters) lies in the first clear_bytes() bytes.
// ---------------------------------------------------------------------------------------------
struct ScratchHdr {
    uint32_t claim;   // dynamic claims taken (claim q = gridDim.x + this counter)
    uint32_t ngen;    // rows listed for the cluster kernel
    uint32_t gclaim;  // listed rows the cluster kernel has claimed
    uint32_t done;    // streaming CTAs that have stopped claiming
};
constexpr int kPartList = 256;  // tokens one segment publishes at most
constexpr int kMaxSegments = 8;  // segments of a split row, at most (a merge parks 32 entries of each)
struct PartHdr {
    float max;       // the segment's maximum (NaN-propagating)
    uint32_t n;      // tokens published
    uint32_t flags;  // PartFlag bits
    uint32_t pad;
};
enum PartFlag : uint32_t { kPartOverflow = 1, kPartTimeout = 2, kPartUnlisted = 4 };
constexpr uint64_t kPartBytes = sizeof(PartHdr) + (uint64_t)kPartList * sizeof(uint64_t);

struct ScratchLayout {
    uint64_t arrive;   // uint32_t[nsplit]: segments of each split row published so far
    uint64_t genlist;  // int32_t[B]: rows left to the cluster kernel
    uint64_t parts;    // nsplit * nseg partials of kPartBytes
    uint64_t total;
    __host__ __device__ static ScratchLayout of(int64_t B, int64_t nsplit, int nseg)
    {
        ScratchLayout L;
        L.arrive = sizeof(ScratchHdr);
        L.genlist = L.arrive + 4ull * (uint64_t)nsplit;
        L.parts = (L.genlist + 4ull * (uint64_t)B + 15ull) & ~15ull;
        L.total = L.parts + (uint64_t)nsplit * (uint64_t)nseg * kPartBytes;
        return L;
    }
    __host__ __device__ uint64_t clear_bytes() const { return genlist; }
};

struct ScratchView {
    ScratchHdr* hdr;
    uint32_t* arrive;
    int32_t* genlist;
    unsigned char* parts;
    __device__ __forceinline__ explicit ScratchView(const Args& a)
    {
        const ScratchLayout L = ScratchLayout::of(a.B, a.nsplit, a.nseg);
        unsigned char* base = static_cast<unsigned char*>(a.scratch);
        hdr = reinterpret_cast<ScratchHdr*>(base);
        arrive = reinterpret_cast<uint32_t*>(base + L.arrive);
        genlist = reinterpret_cast<int32_t*>(base + L.genlist);
        parts = base + L.parts;
    }
    __device__ __forceinline__ PartHdr* part_hdr(int64_t split_row, int seg, int nseg) const
    {
        return reinterpret_cast<PartHdr*>(parts + ((uint64_t)split_row * (uint64_t)nseg + (uint64_t)seg) * kPartBytes);
    }
    __device__ __forceinline__ uint64_t* part_ent(int64_t split_row, int seg, int nseg) const
    {
        return reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(part_hdr(split_row, seg, nseg)) +
                                           sizeof(PartHdr));
    }
};

// Rows left to the cluster kernel in a split batch: sampling with min-p off.  They need the general
// path, which takes several passes over the row: on-chip in the cluster kernel, from global memory
// in the streaming kernel.  (Failed parameters, greedy rows and min-p rows stay with the streaming
// kernel.)
__device__ __forceinline__ bool routed_to_cluster(float T, float P, float MP)
{
    return isfinite(T) && isfinite(P) && isfinite(MP) && T > 0.f && !(MP > 0.f);
}

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
    uint32_t pub_ca;  // exact pass: tokens above the top-p window
    uint64_t pub_z;   // exact pass: fixed-point mass of the survivors
    uint64_t pub_a;   // exact pass: fixed-point mass above the top-p window
    uint32_t pub_claim;  // list mode: the listed row this cluster claimed (rank 0's copy is read)
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
    // --- fine histogram over d of this CTA's survivors (read by the other CTAs): counts in
    //     hc[0, kFineBins), sums of the positions inside the bins (units of 2^-16 bin) after them
    alignas(16) uint32_t hc[2 * kFineBins];
    // --- top-p window: this CTA's exact mass and count per group (read by the other CTAs), and
    //     the cluster's sums
    uint64_t wmass[kMaxWin];
    uint32_t wcnt[kMaxWin];
    uint64_t wm_all[kMaxWin];
    uint32_t wc_all[kMaxWin];
    union alignas(16) {
        struct {  // sub-histogram over a key interval: local, then this CTA's share of the sums
            uint32_t hcnt[kSubBins];
            uint64_t hmass[kSubBins];
            uint32_t rcnt[kSubBins];
            uint64_t rmass[kSubBins];
        } sh;
        struct {  // gathered candidates (key << 32 | ~index), sorted descending, and mass prefixes
            uint64_t sbuf[kCand];
            uint64_t pre[kCand + 1];
        } cd;
        uint32_t rq[kWarps][kRaceQueue];  // race queues: vector index | (token mask << 24)
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
    uint32_t* hr = nullptr;  // cluster-wide fine histogram (2 * kFineBins words, set by the kernel)
    __device__ __forceinline__ uint32_t* fine(Shared&) { return hr; }
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
    __device__ __forceinline__ uint32_t* fine(Shared& s) { return s.hc; }
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
    static constexpr int kEPV = Elem<TIn>::kPerVec;
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
        constexpr int U = kGlobal ? 4 : 1;  // global rows: four loads in flight; shared: short loop body
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

    // Vector by vector with a trip count that is the same for every lane of a warp (a lane past
    // the end gets ok = false), four vectors loaded at a time from global memory: fv(z[kEPV], v,
    // ok); then the ragged elements through fx(z, i).  fv may use warp-wide collectives.
    template <typename FV, typename FX>
    __device__ __forceinline__ void for_each_vec(const Shared& s, FV&& fv, FX&& fx) const
    {
        using E = Elem<TIn>;
        constexpr int U = kGlobal ? 4 : 1;
        const int lane = threadIdx.x & 31;
        for (int vb = (int)threadIdx.x - lane; vb < nvec; vb += U * kThreads) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vb + u * kThreads + lane;
                w[u] = (v < nvec) ? load(v) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vb + u * kThreads + lane;
                float z[kEPV];
                E::unpack(w[u], z);
                fv(z, v, v < nvec);
            }
        }
        for (int x = threadIdx.x; x < s.nx; x += kThreads) fx(s.xz[x], s.xi[x]);
    }
};
template <typename TIn>
using Slice = VecSource<TIn, false>;
template <typename Src>
struct ElemOf;
template <typename TIn, bool kG>
struct ElemOf<VecSource<TIn, kG>> {
    using type = TIn;
};
template <typename TIn>
using GlobalRow = VecSource<TIn, true>;

// NaN-propagating maximum of N floats by a tree of three-input maxima (one instruction each on
// sm_100 and later).
template <int N>
__device__ __forceinline__ float max_tree_nan(const float (&z)[N])
{
    if constexpr (N == 1) {
        return z[0];
    } else if constexpr (N == 2) {
        return fmax_nan(z[0], z[1]);
    } else {
        constexpr int M = (N + 2) / 3;
        float r[M];
#pragma unroll
        for (int i = 0; i < M; ++i) {
            if (3 * i + 2 < N) r[i] = fmax3_nan(z[3 * i], z[3 * i + 1], z[3 * i + 2]);
            else if (3 * i + 1 < N) r[i] = fmax_nan(z[3 * i], z[3 * i + 1]);
            else r[i] = z[3 * i];
        }
        return max_tree_nan(r);
    }
}

// The same over N words of two packed bfloat16 values each (packed maxima, no unpacking).
template <int N>
__device__ __forceinline__ uint32_t bmax_tree_nan(const uint32_t (&x)[N])
{
    if constexpr (N == 1) {
        return x[0];
    } else {
        constexpr int M = (N + 1) / 2;
        uint32_t r[M];
#pragma unroll
        for (int i = 0; i < M; ++i) r[i] = (2 * i + 1 < N) ? bmax2_nan(x[2 * i], x[2 * i + 1]) : x[2 * i];
        return bmax_tree_nan(r);
    }
}

// Maximum (NaN-propagating) over nvec 16-byte vectors, listing every element above thr through
// list(z, i).  Each thread takes kVecs vectors per step and reduces them with a tree of max
// operations -- three-input float maxima for float32, packed bfloat16x2 maxima for bfloat16 (no
// unpacking) -- and only a step whose maximum exceeds thr is looked at element by element, so a pass
// costs well under one instruction per element when little is listed.  The default step is 16
// elements; wider steps measured slower in the streaming kernel (more code in its hot loop).
template <typename TIn, bool kGlobal, int kVecs = 16 / Elem<TIn>::kPerVec, typename ListF>
__device__ __forceinline__ float scan_max_list(const uint4* vec, int nvec, int32_t elem0, float thr, ListF&& list)
{
    using E = Elem<TIn>;
    constexpr int EPV = E::kPerVec;
    constexpr int U = kVecs;  // vectors per step
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
        float m;
        if constexpr (EPV == 4) {
            float z[4 * U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                z[4 * u] = __uint_as_float(w[u].x);
                z[4 * u + 1] = __uint_as_float(w[u].y);
                z[4 * u + 2] = __uint_as_float(w[u].z);
                z[4 * u + 3] = __uint_as_float(w[u].w);
            }
            m = max_tree_nan(z);
        } else {
            uint32_t x[4 * U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                x[4 * u] = w[u].x;
                x[4 * u + 1] = w[u].y;
                x[4 * u + 2] = w[u].z;
                x[4 * u + 3] = w[u].w;
            }
            const uint32_t c = bmax_tree_nan(x);
            m = fmax_nan(__uint_as_float(c << 16), __uint_as_float(c & 0xFFFF0000u));
        }
        cm = fmax_nan(cm, m);
        if (m > thr) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float t[EPV];
                E::unpack(w[u], t);
#pragma unroll
                for (int j = 0; j < EPV; ++j)
                    if (t[j] > thr) list(t[j], elem0 + (v + u * kThreads) * EPV + j);
            }
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

// Fine bin of a scaled distance d32 >= 0: floor(min(d32, kFineBins - 1)), with float adds only.
// For every integer 1 <= b <= kFineBins - 1:  fine_bin(d32) < b  <=>  d32 < b.
__device__ __forceinline__ int fine_bin(float d32)
{
    const float c = fminf(d32, (float)(kFineBins - 1));
    return (int)(__float_as_uint(__fadd_rd(c, 0x1p23f)) - 0x4B000000u);
}

// Position of d32 inside its bin b (b <= d32 < b + 1, so d32 - b is exact) in units of 2^-16,
// rounded to nearest: 0 .. 65536.
__device__ __forceinline__ uint32_t bin_pos16(float d32, int b)
{
    return __float_as_uint(__fmaf_rn(d32 - (float)b, 65536.f, 0x1p23f)) - 0x4B000000u;
}

// Whether a scaled distance d32 falls in the fine bins [b_lo, b_end).  The last bin has no upper
// bound: it holds every d32 >= kFineBins - 1, including +inf (a temperature small enough to overflow
// (zmax - z) / T), so ranges are always tested through fine_bin, never against a float bound.
__device__ __forceinline__ bool in_bins(float d32, int b_lo, int b_end)
{
    const int b = fine_bin(d32);
    return b >= b_lo && b < b_end;
}

// Cluster-wide sum of the CTAs' fine histograms hc into hr (a copy for a cluster of one CTA; nothing
// to do when hr is hc itself).
// Starts with a topology barrier: every CTA's histogram and published values are then complete,
// and stay readable until the caller's next topology barrier.
template <typename Topo>
__device__ __forceinline__ void reduce_fine(Topo& topo, Shared& s, uint32_t* hr)
{
    topo.sync();
    if (topo.C > 1) {
        for (int v = threadIdx.x; v < 2 * kFineBins / 4; v += kThreads) {
            uint4 acc = make_uint4(0u, 0u, 0u, 0u);
            for (uint32_t q = 0; q < topo.C; ++q) {
                const uint4 x = *reinterpret_cast<const uint4*>(topo.map(&s.hc[4 * v], q));
                acc.x += x.x;
                acc.y += x.y;
                acc.z += x.z;
                acc.w += x.w;
            }
            reinterpret_cast<uint4*>(hr)[v] = acc;
        }
        cta_sync();
    } else if (hr != s.hc) {  // a cluster of one CTA keeps its sums apart like a wider one
        for (int v = threadIdx.x; v < 2 * kFineBins / 4; v += kThreads)
            reinterpret_cast<uint4*>(hr)[v] = reinterpret_cast<const uint4*>(s.hc)[v];
        cta_sync();
    }
}

// Top-k on the fine counts: the last non-empty bin b with (count above b) < K, and that count.
// Thread t owns bins 2t and 2t+1 (kFineBins == 2 * kThreads).
__device__ __forceinline__ void fine_scan_topk(Shared& s, const uint32_t* hr, uint64_t K, int* out_b, uint64_t* out_c)
{
    const int t = threadIdx.x;
    const uint2 c2 = reinterpret_cast<const uint2*>(hr)[t];
    const uint32_t c[2] = {c2.x, c2.y};
    uint64_t tot;
    const uint64_t pre = block_exscan_u64((uint64_t)c2.x + c2.y, s, &tot);
    uint32_t best = 0;
    uint64_t cum = pre, at = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (c[j] > 0 && cum < K) {
            best = (uint32_t)(2 * t + j) + 1u;
            at = cum;
        }
        cum += c[j];
    }
    const uint32_t bb = block_max_u32(best, s);  // >= 1: the bin of the maximum has nothing above it
    if (bb != 0 && best == bb) s.b64[0] = at;
    cta_sync();
    *out_b = (int)bb - 1;
    *out_c = s.b64[0];
    cta_sync();
}

// The bins of d where the top-p crossing can lie, from the fine histogram alone.  A token of bin b
// has d = (b + t) / 16 with t in [0, 1); its mass e^-d lies between (convexity of e^-x) the tangent
// value at the bin's mean position and the chord across the bin:
//   n e^-b/16 e^-mean(t)/16  <=  sum over the bin  <=  n e^-b/16 (1 - (1 - e^-1/16) mean(t)),
// a relative gap below 5e-4.  mean(t) comes from the summed positions (to 2^-17 per token; a bin
// with 65536 or more tokens, or the partial bin bk, uses t in [0, 1]; the last bin [0, e^-511/16]).
// Margins of 4e-6 relative and one unit per token cover expf's error and the fixed-point rounding,
// and the bounds are summed as exact 64-bit fixed-point integers.  With the mass above bin b within
// [cum_lo(b), cum_hi(b)] and Z within [Zlo, Zhi], the crossing (the last bin whose mass above is
// below P Z) is a bin b with cum_lo(b) < P Zhi and cum_hi(b+1) >= P Zlo; every bin before the first
// such bin is certainly kept.  c_b = counts of S: hr[b] below bk, `part` at bk, 0 above.  The
// window's bins form at most kMaxWin groups of 2^sh bins; `list` is set when the window and
// everything above it hold at most kCand tokens.
struct Window {
    int b_lo, b_end, sh, nw;
    bool list;
};
__device__ __forceinline__ Window top_p_window(Shared& s, const uint32_t* hr, int bk, uint32_t part, float P)
{
    const int t = threadIdx.x;
    const float kChord = 1.f - expf(-1.f / kFineScale);
    uint32_t c[2];
    uint64_t lo[2], hi[2];
    uint32_t last = 0;  // 1 + the last non-empty bin of this thread
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int b = 2 * t + j;
        const uint32_t n = (b < bk) ? hr[b] : (b == bk ? part : 0u);
        c[j] = n;
        lo[j] = hi[j] = 0;
        if (n == 0) continue;
        last = (uint32_t)b + 1u;
        const float eb = expf(-(float)b * (1.f / kFineScale));
        float mlo = 0.f, mhi = 1.f;  // bounds of the mean position
        if (b < bk && b < kFineBins - 1 && n < 65536u) {
            const float F = (float)hr[kFineBins + b], nf = (float)n;
            mlo = fmaxf(0.f, (F - 0.5f * nf) / (65536.f * nf) - 1e-6f);
            mhi = fminf(1.f, (F + 0.5f * nf) / (65536.f * nf) + 1e-6f);
        }
        float el = 0.f, eh;
        if (b < kFineBins - 1) {
            el = eb * expf(-mhi * (1.f / kFineScale)) * (1.f - 4e-6f);
            eh = eb * (1.f - kChord * mlo) * (1.f + 4e-6f);
        } else {
            eh = eb * (1.f + 4e-6f);
        }
        const uint64_t ql = fixed44(fminf(el, 1.f)), qh = fixed44(fminf(eh, 1.f));
        lo[j] = (uint64_t)n * (ql > 0 ? ql - 1 : 0);
        hi[j] = (uint64_t)n * (qh + 1);
    }
    uint64_t Zlo, Zhi;
    const uint64_t plo = block_exscan_u64(lo[0] + lo[1], s, &Zlo);
    const uint64_t phi = block_exscan_u64(hi[0] + hi[1], s, &Zhi);
    const double tlo = (double)P * (double)Zlo, thi = (double)P * (double)Zhi;
    uint32_t b0 = (uint32_t)kFineBins, b1 = 0;
    uint64_t cl = plo, ch = phi;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t b = (uint32_t)(2 * t + j);
        if ((double)cl < thi) b1 = b;
        cl += lo[j];
        ch += hi[j];
        if ((double)ch >= tlo && b0 == (uint32_t)kFineBins) b0 = b;
    }
    b0 = block_min_u32(b0, s);
    b1 = block_max_u32(b1, s);
    const uint32_t lastb = block_max_u32(last, s);  // >= 1
    if (b0 >= (uint32_t)kFineBins) b0 = 0;          // cannot happen with P < 1; keep a valid window
    b1 = min(b1, lastb - 1u);
    if (b1 < b0) b1 = b0;
    uint32_t upto = 0;  // tokens of S in bins <= b1
#pragma unroll
    for (int j = 0; j < 2; ++j)
        if ((uint32_t)(2 * t + j) <= b1) upto += c[j];
    upto = block_sum_u32(upto, s);
    Window w;
    w.b_lo = (int)b0;
    w.b_end = (int)b1 + 1;
    const int nb = w.b_end - w.b_lo;
    w.sh = 0;
    while (((nb - 1) >> w.sh) + 1 > kMaxWin) ++w.sh;
    w.nw = ((nb - 1) >> w.sh) + 1;
    w.list = upto <= (uint32_t)kCand;
    return w;
}

// Cluster-wide sum of the sub-histogram u.sh.hcnt/hmass[0, nb) into u.sh.hcnt/hmass of every CTA.
// Step 1: CTA c sums its share of the bins over all CTAs (one remote read per thread) into
// u.sh.rcnt/rmass; step 2: every CTA copies all shares back into its own hcnt/hmass.
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
        const uint32_t c = *topo.map(&s.u.sh.hcnt[b], r);
        if (c) {
            atomicAdd(&s.u.sh.rcnt[b], c);
            atomicAdd((unsigned long long*)&s.u.sh.rmass[b], (unsigned long long)*topo.map(&s.u.sh.hmass[b], r));
        }
    }
    topo.sync();  // all shares complete; nobody reads another CTA's hcnt/hmass any more
    for (int b = threadIdx.x; b < nb; b += kThreads) {
        const uint32_t owner = (uint32_t)(b / per);
        s.u.sh.hcnt[b] = *topo.map(&s.u.sh.rcnt[b], owner);
        s.u.sh.hmass[b] = *topo.map(&s.u.sh.rmass[b], owner);
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

// Scan the (full) sub-histogram u.sh.hcnt/hmass[0, nb) from bin 0 (largest logits) down and return the
// last non-empty bin whose (count, mass) above satisfies the criterion.  nb <= kThreads.
__device__ __forceinline__ void scan_bins(Shared& s, int nb, const Crit& cr, uint64_t C0, uint64_t A0,
                                          int* out_bin, uint64_t* out_c, uint64_t* out_a)
{
    const int b = threadIdx.x;
    const uint64_t c = (b < nb) ? s.u.sh.hcnt[b] : 0;
    const uint64_t m = (b < nb) ? s.u.sh.hmass[b] : 0;
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

// Copy every CTA's candidate list (counts in pub_gcnt) into u.cd.sbuf (unsorted).  Returns n.
template <typename Topo>
__device__ __forceinline__ int gather_lists(Topo& topo, Shared& s)
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
    return (int)n;
}

template <typename Topo>
__device__ __forceinline__ int gather_and_sort(Topo& topo, Shared& s)
{
    const int n = gather_lists(topo, s);
    block_sort_desc(s, n);
    return n;
}

// Race key in float (for pruning) and in double (for the decision) of kept token i.
struct RaceCtx {
    uint32_t k0, k1;    // Philox key = seed
    uint32_t row, s_lo, s_hi;
};

__device__ __forceinline__ float race_u(const RaceCtx& rc, int32_t i)
{
    const uint4 x = philox_block(make_uint4((uint32_t)i >> 2, rc.row, rc.s_lo, rc.s_hi), rc.k0, rc.k1);
    return (float)uniform_grid(pick_word(x, (uint32_t)i & 3u)) * 0x1p-24f;
}

__device__ __forceinline__ float race_key32(float d, float u) { return -d - logf(-logf(u)); }

// The race key in double precision (the float64 definition), out of line: only near-ties need it.
static __device__ __noinline__ double race_key64_(float zmax, float T, float z, float u)
{
    const double d = __ddiv_rn(__dsub_rn((double)zmax, (double)z), (double)T);
    const double g = log(-log((double)u));
    return __dsub_rn(-d, g);
}
__device__ __forceinline__ double race_key64(const RowCtx& r, float z, float u) { return race_key64_(r.zmax, r.T, z, u); }

// Margin between the float race key and the double one (both tokens' errors), for a row whose
// kept tokens have d <= dcut.
__device__ __forceinline__ float race_tol(float dcut) { return 1e-5f + 1e-6f * dcut; }

// Refine the cut among the survivors (min-p, key >= key_lo) whose scaled distance d32 lies in the
// fine bins [b_lo, b_end), given the (count, mass) of the survivors above that range.  Exact: ends
// with a sorted candidate list or with a single logit value.  Starts with a topology barrier.
// Each round is one pass over the row: the survivors of the current key interval are counted,
// listed (the first kCand) and histogrammed over kSubBins sub-intervals at once; a round with at
// most kCand of them sorts the list (or finds a single class), otherwise the crossing sub-interval
// becomes the next interval.  The first interval holds every logit whose distance can fall in the
// fine bins (their bounds widened by a relative 1e-5, far above the float rounding of the
// distance); the bin test itself stays exact.  Lanes of a warp holding the same key (a tie class)
// add to the histogram once, together: a class of thousands of tied logits would otherwise queue
// on one shared-memory address.  need_mass = false (a count criterion whose caller uses only the
// key and the count) skips the fixed-point mass sums.
template <typename Topo, typename Src>
__device__ Sel refine_range(Topo& topo, Shared& s, const Src& sl, const RowCtx& r, float zc, int b_lo, int b_end,
                            uint32_t key_lo, const Crit& cr, uint64_t C0, uint64_t A0, bool need_mass = true)
{
    const uint32_t C = topo.C;
    uint32_t klo, khi;
    {
        const float w_lo = (float)b_lo * (r.T / kFineScale), w_hi = (float)b_end * (r.T / kFineScale);
        const float slack = 1e-5f * (fabsf(r.zmax) + w_hi) + 1e-30f;
        khi = fkey(r.zmax - w_lo + slack);
        klo = (b_end >= kFineBins) ? 0u : fkey(r.zmax - w_hi - slack);
        if (!(isfinite(w_hi) && isfinite(slack))) klo = 0u;  // huge T: no useful lower bound
        if (!isfinite(r.zmax - w_lo + slack)) khi = 0xFFFFFFFFu;
        klo = max(klo, key_lo);
    }
    bool by_range = true;
    for (int iter = 0; iter < 8; ++iter) {
        topo.sync();  // nobody still reads my candidate list, published counts or shares
        int sh = 0;
        while (khi >= klo && ((uint64_t)(khi - klo) >> sh) >= (uint64_t)kSubBins) ++sh;
        const int nsub = (khi >= klo) ? (int)((uint64_t)(khi - klo) >> sh) + 1 : 1;
        for (int b = threadIdx.x; b < kSubBins; b += kThreads) {
            s.u.sh.hcnt[b] = 0;
            s.u.sh.hmass[b] = 0;
        }
        if (threadIdx.x == 0) s.ncand = 0;
        cta_sync();
        uint32_t lcnt = 0, lmin = 0xFFFFFFFFu, lmax = 0;
        const uint32_t lo = klo, hi = khi;
        sl.for_each(s, [&](float z, int32_t i) {
            if (!(z > zc)) return;
            const uint32_t key = fkey(z);
            if (key < key_lo || key < lo || key > hi) return;
            const float d = dist(r, z);
            if (by_range && !in_bins(d * kFineScale, b_lo, b_end)) return;
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
            const uint32_t peers = __match_any_sync(__activemask(), key);  // this warp's lanes with this key
            if ((threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1)) {
                const uint32_t np = (uint32_t)__popc(peers);
                const int sb = (int)((hi - key) >> sh);
                atomicAdd(&s.u.sh.hcnt[sb], np);
                if (need_mass)
                    atomicAdd((unsigned long long*)&s.u.sh.hmass[sb], (unsigned long long)np * qmass_d(d));
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
        // Too many: the sub-interval holding the crossing (sub-bin 0 = largest keys) is next.
        cluster_reduce_hist(topo, s, kSubBins);
        int jb;
        uint64_t c_at, a_at;
        scan_bins(s, nsub, cr, C0, A0, &jb, &c_at, &a_at);
        if (jb < 0) jb = 0;
        C0 = c_at;
        A0 = a_at;
        const uint64_t top = (uint64_t)hi - ((uint64_t)jb << sh);
        const uint64_t width = (uint64_t)1 << sh;
        const uint64_t bot = (top + 1 >= width) ? top + 1 - width : 0;
        khi = (uint32_t)min(top, (uint64_t)gmax);
        klo = (uint32_t)max((uint64_t)max(lo, gmin), bot);
        by_range = false;
    }
    // Unreachable in practice (each round shrinks the 32-bit interval by 2^7); keep a valid answer.
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
// z_ext != 0: the list is the top of a larger set whose fixed-point mass is z_ext (top-p is taken
// against it; top-k must then be off).
// The sorted survivors are left in buf[0, n) (descending).
__device__ __forceinline__ WarpResult warp_resolve(uint64_t* buf, const RowCtx& r, const RaceCtx& rc, uint32_t n,
                                                   bool topk_on, int32_t K, float P, uint64_t z_ext = 0)
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
    __syncwarp();  // every lane has read its entry of buf
    if (lane < n) buf[lane] = v;
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
    uint64_t zs = z_ext ? z_ext : total;
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
// then the race.  For the scan and the cuts lane l owns sorted positions [8 l, 8 l + 8); the masses
// and the race's Philox draws are spread over all lanes (position l + 32 m), so a list of a few dozen
// survivors does not leave most lanes idle.  Every lane returns the same result.
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
    // masses at strided positions (every lane busy), parked in pre[] for the scan below
    for (uint32_t pos = lane; pos < n; pos += 32) pre[pos] = qmass_d(dist(r, key_to_float(sb_key(sorted[pos]))));
    __syncwarp();
    const uint32_t p0 = 8 * lane;
    uint64_t q[8];
    uint32_t kk[8];
    uint64_t loc = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t pos = p0 + m;
        kk[m] = (pos < n) ? sb_key(sorted[pos]) : 0u;
        q[m] = (pos < n) ? pre[pos] : 0;
        loc += q[m];
    }
    __syncwarp();  // every lane has read its masses before pre[] is overwritten with prefixes
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
    // race over positions < nk, strided over the lanes (position lane + 32 m) so every lane draws
    float k32[8], uu[8];
    float m32 = -INFINITY;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t pos = lane + 32u * (uint32_t)m;
        k32[m] = -INFINITY;
        uu[m] = 0.f;
        if (pos < nk) {
            const uint64_t v = sorted[pos];
            uu[m] = race_u(rc, sb_idx(v));
            k32[m] = race_key32(dist(r, key_to_float(sb_key(v))), uu[m]);
            m32 = fmaxf(m32, k32[m]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m32 = fmaxf(m32, __shfl_xor_sync(0xFFFFFFFFu, m32, o));
    const float tol = race_tol(dist(r, key_to_float(key_cut)));
    uint32_t nf = 0, fpos = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t pos = lane + 32u * (uint32_t)m;
        if (pos < nk && k32[m] >= m32 - tol) {
            ++nf;
            fpos = pos;
        }
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
            const uint32_t pos = lane + 32u * (uint32_t)m;
            if (pos < nk && k32[m] >= m32 - tol) {
                const uint64_t v = sorted[pos];
                const double k64 = race_key64(r, key_to_float(sb_key(v)), uu[m]);
                const int32_t i = sb_idx(v);
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
// race.  n <= 32 runs in warp 0 alone; larger n sorts with the whole CTA.  z_ext != 0: the list is
// the top of the survivors, whose whole fixed-point mass is z_ext (top-k already applied).
__device__ __forceinline__ RowResult resolve_candidates(Shared& s, const RowCtx& r, const RaceCtx& rc, uint32_t n,
                                                        bool topk_on, int32_t K, float P, uint64_t z_ext = 0)
{
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    RowResult out;
    if (n <= 32) {
        if (tid < 32) {
            const WarpResult wr = warp_resolve(s.u.cd.sbuf, r, rc, n, topk_on, K, P, z_ext);
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
    uint64_t ZS = z_ext ? z_ext : s.u.cd.pre[n];
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

// Per-thread race over kept tokens: the best two float race keys (and the best's index).  A token
// is skipped without drawing its uniform when even the largest -ln(-ln u) of the uniform grid
// (u = 1 - 2^-24 gives 16.6355...) cannot lift its key to this thread's second-best key: such a
// token can be neither the best nor the second best.  Consecutive tokens share one Philox block.
struct RaceAcc {
    Top2 t2;
    uint32_t ctr;
    uint4 x;
    __device__ __forceinline__ void init()
    {
        t2.init();
        ctr = 0xFFFFFFFFu;
    }
    __device__ __forceinline__ void add(const RaceCtx& rc, float d, int32_t i)
    {
        if (16.64f - d < t2.k2) return;
        const uint32_t c = (uint32_t)i >> 2;
        if (c != ctr) {
            ctr = c;
            x = philox_block(make_uint4(c, rc.row, rc.s_lo, rc.s_hi), rc.k0, rc.k1);
        }
        const float u = (float)uniform_grid(pick_word(x, (uint32_t)i & 3u)) * 0x1p-24f;
        t2.add(race_key32(d, u), i);
    }
};

// Per-warp queue of vectors holding tokens to race, so that the Philox blocks and logarithms run
// for full warps: a lane queues (vector, token mask) when it finds tokens to race, and every 64
// queued vectors are raced two per lane, the first Philox block of each pair drawn together.  Any
// lane may race any token: a token skipped against some lane's second-best key cannot be among the
// two best of the row.
template <typename Src>
struct RaceQueue {
    uint32_t* q;  // this warp's kRaceQueue entries: vector | (mask << 24)
    uint32_t n;   // queued entries (the same in every lane)
    __device__ __forceinline__ explicit RaceQueue(Shared& s) : q(s.u.rq[threadIdx.x >> 5]), n(0) {}
    __device__ __forceinline__ void race_vector(const Src& src, const RowCtx& r, const RaceCtx& rc, RaceAcc& race,
                                                uint32_t e, uint4 x)
    {
        const int v = (int)(e & 0xFFFFFFu);
        const uint32_t mask = e >> 24;
        float z[Src::kEPV];
        Elem<typename ElemOf<Src>::type>::unpack(src.load(v), z);
        const int32_t i0 = (int32_t)src.elem0 + v * Src::kEPV;
        race.ctr = (uint32_t)i0 >> 2;  // the block of the vector's first token, drawn by the caller
        race.x = x;
#pragma unroll
        for (int j = 0; j < Src::kEPV; ++j)
            if ((mask >> j) & 1u) race.add(rc, dist(r, z[j]), i0 + j);
    }
    // Races entries [0, cnt) (cnt <= 64): lane l takes entries l and l + 32.
    __device__ __forceinline__ void run(const Src& src, const RowCtx& r, const RaceCtx& rc, RaceAcc& race, uint32_t cnt)
    {
        const uint32_t lane = threadIdx.x & 31;
        if (lane >= cnt) return;
        const uint32_t e0 = q[lane];
        const bool two = lane + 32u < cnt;
        const uint32_t e1 = two ? q[lane + 32u] : e0;
        const uint32_t c0 = (uint32_t)((int32_t)src.elem0 + (int)(e0 & 0xFFFFFFu) * Src::kEPV) >> 2;
        const uint32_t c1 = (uint32_t)((int32_t)src.elem0 + (int)(e1 & 0xFFFFFFu) * Src::kEPV) >> 2;
        uint4 x0 = make_uint4(c0, rc.row, rc.s_lo, rc.s_hi), x1 = make_uint4(c1, rc.row, rc.s_lo, rc.s_hi);
        philox4x32_10_x2(x0, x1, rc.k0, rc.k1);
        race_vector(src, r, rc, race, e0, x0);
        if (two) race_vector(src, r, rc, race, e1, x1);
    }
    // Every lane calls this for its vector v (mask 0: nothing to race).
    __device__ __forceinline__ void push(const Src& src, const RowCtx& r, const RaceCtx& rc, RaceAcc& race, int v,
                                         uint32_t mask)
    {
        const uint32_t lane = threadIdx.x & 31;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, mask != 0u);
        if (bal == 0u) return;
        if (mask) q[n + __popc(bal & ((1u << lane) - 1u))] = (uint32_t)v | (mask << 24);
        n += __popc(bal);
        if (n >= 64u) {  // at most 63 + 32 < kRaceQueue entries
            __syncwarp();
            run(src, r, rc, race, 64u);
            __syncwarp();
            if (lane + 64u < n) q[lane] = q[lane + 64u];
            __syncwarp();
            n -= 64u;
        }
    }
    __device__ __forceinline__ void drain(const Src& src, const RowCtx& r, const RaceCtx& rc, RaceAcc& race)
    {
        __syncwarp();
        run(src, r, rc, race, n);
        __syncwarp();
        n = 0;
    }
};

// Merge the threads' race results over the topology and decide the token exactly: the best float
// key wins when it leads the second by more than the float/double margin; otherwise every kept
// token (key >= kc) within the margin of the best is re-evaluated in double precision.
template <typename Topo, typename Src>
__device__ int32_t race_finish(Topo& topo, Shared& s, const Src& src, const RowCtx& r, const RaceCtx& rc, Top2 t2,
                               uint32_t kc)
{
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    const uint32_t C = topo.C;
    const float tol = race_tol(dist(r, key_to_float(kc)));
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
    int32_t token = (int32_t)s.bu[6];
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
        token = (int32_t)s.bu[6];
    }
    cta_sync();
    return token;
}

// Sum of one u64 per thread over the CTA (every thread gets it).
__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, Shared& s)
{
    uint64_t tot;
    (void)block_exscan_u64(v, s, &tot);
    return tot;
}

// The general path, for rows whose survivors are not already listed.  S0 = the min-p survivors
// against the global maximum (z > zc and minp_ok); S = S0 cut by top-k; the kept set = S cut by
// top-p.  Every cut is an upper set in z, found exactly:
//   A. one pass: counts of S0 over fine bins of d (32-bit atomics), the first kCand listed;
//      few survivors -> sort the lists and resolve them;
//   B. top-k from the counts, refined exactly inside its crossing bin (or, when everything down to
//      that bin fits a list, by listing it);
//   C. top-p: bounds on the bins' masses give a window of bins holding the crossing; one exact
//      pass sums the fixed-point masses of S (per thread, no atomics), of the tokens above the
//      window, and per window group (atomics on window tokens only), racing the tokens above the
//      window, which are certainly kept; then an exact refinement inside the crossing group and
//      a race over the window's kept tokens.  A window that does not hold the crossing (not
//      expected: the bounds are rigorous) is replaced by one covering every bin.
// Starts with a topology barrier, so the caller's published values may still be read by other CTAs
// when it is entered.
template <typename Topo, typename Src>
__device__ RowResult general_path(Topo& topo, Shared& s, const Src& src, const RowCtx& r, float zc, bool topk_on,
                                  int32_t K, float P, const RaceCtx& rc, float* prow, bool need_zk = false)
{
    const int tid = threadIdx.x;
    const uint32_t lane = tid & 31;
    const uint32_t C = topo.C;
    uint32_t* hr = topo.fine(s);

    // ---- A: fine counts of S0, the first kCand survivors listed
    topo.sync();  // nobody still reads the caller's lists or published values
    for (int b = tid; b < 2 * kFineBins; b += kThreads) s.hc[b] = 0;
    if (tid == 0) s.ncand = 0;
    cta_sync();
    uint32_t my_minkey = 0xFFFFFFFFu;
    bool full = false;
    src.for_each(s, [&](float z, int32_t i) {
        if (!(z > zc)) return;
        const float d = dist(r, z);
        if (!minp_ok(r, z, d)) return;
        const uint32_t key = fkey(z);
        my_minkey = min(my_minkey, key);
        const float d32 = d * kFineScale;
        const int b = fine_bin(d32);
        atomicAdd(&s.hc[b], 1u);
        if (b < kFineBins - 1) atomicAdd(&s.hc[kFineBins + b], bin_pos16(d32, b));
        if (!full) {
            const uint32_t slot = atomicAdd(&s.ncand, 1u);
            if (slot < (uint32_t)kCand) {
                s.ckey[slot] = key;
                s.cidx[slot] = (uint32_t)i;
            } else {
                full = true;
            }
        }
    });
    my_minkey = block_min_u32(my_minkey, s);
    if (tid == 0) {
        s.pub_gcnt = min(s.ncand, (uint32_t)kCand);
        s.pub_minkey = my_minkey;
    }
    reduce_fine(topo, s, hr);  // topology barrier first
    if (tid < 32) {
        uint32_t mk = (lane < C) ? *topo.map(&s.pub_minkey, lane) : 0xFFFFFFFFu;
        mk = warp_min_u32(mk);
        if (lane == 0) s.bu[3] = mk;
    }
    uint32_t ns0 = 0;
    {
        const uint2 c2 = reinterpret_cast<const uint2*>(hr)[tid];
        ns0 = block_sum_u32(c2.x + c2.y, s);  // (its barriers publish bu[3])
    }
    const uint32_t min_key = s.bu[3];
    RowResult res;

    if (ns0 <= (uint32_t)kCand) {
        // ---- few survivors: every one is on some CTA's list
        const int n = gather_lists(topo, s);
        res = resolve_candidates(s, r, rc, (uint32_t)n, topk_on, K, P);
        if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
        return res;
    }

    // ---- B: top-k on the counts
    uint32_t key_k = 0;
    uint64_t NS = ns0;
    int bk = kFineBins;  // bins above bk hold no token of S; bin bk holds `part` of them
    uint32_t part = 0;
    if (topk_on && (uint64_t)ns0 > (uint64_t)K) {
        uint64_t ck;
        fine_scan_topk(s, hr, (uint64_t)K, &bk, &ck);
        const uint64_t upto = ck + hr[bk];
        if (upto <= (uint64_t)kCand) {
            // everything down to the crossing bin fits one list: list it and resolve exactly
            topo.sync();  // the other CTAs are done with this CTA's published values
            if (tid == 0) s.ncand = 0;
            cta_sync();
            src.for_each(s, [&](float z, int32_t i) {
                if (!(z > zc)) return;
                const float d = dist(r, z);
                if (fine_bin(d * kFineScale) > bk || !minp_ok(r, z, d)) return;
                const uint32_t slot = atomicAdd(&s.ncand, 1u);
                s.ckey[slot] = fkey(z);
                s.cidx[slot] = (uint32_t)i;
            });
            cta_sync();
            if (tid == 0) s.pub_gcnt = s.ncand;
            topo.sync();
            const int n = gather_lists(topo, s);
            res = resolve_candidates(s, r, rc, (uint32_t)n, topk_on, K, P);
            if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
            return res;
        }
        Crit ck2;
        ck2.by_mass = false;
        ck2.tcnt = (uint64_t)K;
        ck2.tmass = 0.0;
        const Sel sk = refine_range(topo, s, src, r, zc, bk, bk + 1, 0u, ck2, ck, 0, false);
        key_k = sk.key;
        NS = sk.cnt;
        part = (uint32_t)(sk.cnt - ck);
    }

    // ---- C: top-p and the race
    RaceAcc race;
    race.init();
    if (!(P > 0.f && P < 1.f)) {
        if (P <= 0.f) {  // only the top class
            Crit c1;
            c1.by_mass = false;
            c1.tcnt = 1;
            c1.tmass = 0.0;
            const Sel s1 = refine_range(topo, s, src, r, zc, 0, 1, key_k, c1, 0, 0);
            res.key_cut = s1.key;
            res.nk = s1.cnt;
            res.zk = s1.mass;
        } else {  // no top-p cut: S is kept
            res.key_cut = max(key_k, min_key);
            res.nk = NS;
            res.zk = 0;
        }
        const uint32_t kc = res.key_cut;
        const bool sum_z = (prow != nullptr || need_zk) && P >= 1.f;  // the kept mass (probabilities, log-probability)
        uint64_t zhi = 0, zlo = 0;
        RaceQueue<Src> rq(s);
        auto kept = [&](float z) -> bool {  // kept; sums its mass when asked; true if it may race
            if (!((z > -INFINITY) && fkey(z) >= kc)) return false;
            const float d = dist(r, z);
            if (sum_z) {
                const Fixed44 f = fixed44_parts(expf(-d));
                zhi += f.hi;
                zlo += f.lo;
            }
            return !(16.64f - d < race.t2.k2);
        };
        src.for_each_vec(
            s,
            [&](const float* z, int v, bool ok) {
                uint32_t mask = 0;
                if (ok)
#pragma unroll
                    for (int j = 0; j < Src::kEPV; ++j)
                        if (kept(z[j])) mask |= 1u << j;
                rq.push(src, r, rc, race, v, mask);
            },
            [&](float z, int32_t i) {
                if (kept(z)) race.add(rc, dist(r, z), i);
            });
        rq.drain(src, r, rc, race);
        if (sum_z) {
            const uint64_t cta = block_sum_u64((zhi << 22) + zlo, s);
            if (tid == 0) s.pub_z = cta;
            topo.sync();
            if (tid < 32) {
                uint64_t z = (lane < C) ? *topo.map(&s.pub_z, lane) : 0;
                z = warp_sum_u64(z);
                if (lane == 0) s.b64[2] = z;
            }
            cta_sync();
            res.zk = s.b64[2];
        }
        res.token = race_finish(topo, s, src, r, rc, race.t2, kc);
        if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
        return res;
    }

    Window w = top_p_window(s, hr, bk, part, P);
    uint64_t Z = 0, A = 0;
    uint32_t CA = 0;
    double tmass = 0.0;
    int nlist = -1;  // list mode: the sorted list of S down to the window's end
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (attempt == 1) {  // a window covering every bin
            w.b_lo = 0;
            w.b_end = kFineBins;
            w.sh = 0;
            while (((kFineBins - 1) >> w.sh) + 1 > kMaxWin) ++w.sh;
            w.nw = ((kFineBins - 1) >> w.sh) + 1;
            w.list = false;
            race.init();
        }
        // window bins [b_lo, b_end); a window reaching the last bin has no upper bound (d = +inf included)
        const float flo = (float)w.b_lo;
        const bool open_end = w.b_end >= kFineBins;
        const float fend = open_end ? INFINITY : (float)w.b_end;
        const bool list = w.list;
        const int b_lo = w.b_lo, sh = w.sh;
        topo.sync();  // nobody still reads this CTA's window sums, lists or published values
        if (tid < kMaxWin) {
            s.wmass[tid] = 0;
            s.wcnt[tid] = 0;
        }
        if (tid == 0) s.ncand = 0;
        cta_sync();
        uint64_t zhi = 0, zlo = 0, ahi = 0, alo = 0;  // high (x 2^22) and low parts of the sums
        uint32_t ca = 0;
        RaceQueue<Src> rq(s);
        // sums for one token; true when it is certainly kept and may race
        auto one = [&](float z, int32_t i) -> bool {
            if (!(z > zc)) return false;
            const uint32_t key = fkey(z);
            if (key < key_k) return false;
            const float d = dist(r, z);
            if (!minp_ok(r, z, d)) return false;
            const Fixed44 f = fixed44_parts(expf(-d));
            zhi += f.hi;
            zlo += f.lo;
            const float d32 = d * kFineScale;
            if (list) {
                if (open_end || d32 < fend) {
                    const uint32_t slot = atomicAdd(&s.ncand, 1u);
                    s.ckey[slot] = key;
                    s.cidx[slot] = (uint32_t)i;
                }
                return false;
            }
            if (d32 < flo) {  // certainly kept
                ahi += f.hi;
                alo += f.lo;
                ++ca;
                return !(16.64f - d < race.t2.k2);
            }
            if (open_end || d32 < fend) {
                const int g = (fine_bin(d32) - b_lo) >> sh;
                atomicAdd((unsigned long long*)&s.wmass[g], (unsigned long long)(((uint64_t)f.hi << 22) + f.lo));
                atomicAdd(&s.wcnt[g], 1u);
            }
            return false;
        };
        src.for_each_vec(
            s,
            [&](const float* z, int v, bool ok) {
                uint32_t mask = 0;
                if (ok) {
                    const int32_t i0 = (int32_t)src.elem0 + v * Src::kEPV;
#pragma unroll
                    for (int j = 0; j < Src::kEPV; ++j)
                        if (one(z[j], i0 + j)) mask |= 1u << j;
                }
                rq.push(src, r, rc, race, v, mask);
            },
            [&](float z, int32_t i) {
                if (one(z, i)) race.add(rc, dist(r, z), i);
            });
        rq.drain(src, r, rc, race);
        const uint64_t zc_ = block_sum_u64((zhi << 22) + zlo, s);
        const uint64_t ac_ = block_sum_u64((ahi << 22) + alo, s);
        const uint32_t cc_ = block_sum_u32(ca, s);
        if (tid == 0) {
            s.pub_z = zc_;
            s.pub_a = ac_;
            s.pub_ca = cc_;
            s.pub_gcnt = s.ncand;
        }
        topo.sync();
        if (tid < 32) {
            uint64_t z = 0, a = 0;
            uint32_t c = 0;
            if (lane < C) {
                z = *topo.map(&s.pub_z, lane);
                a = *topo.map(&s.pub_a, lane);
                c = *topo.map(&s.pub_ca, lane);
            }
            z = warp_sum_u64(z);
            a = warp_sum_u64(a);
            c = warp_sum_u32(c);
            if (lane == 0) {
                s.b64[2] = z;
                s.b64[3] = a;
                s.bu[7] = c;
            }
        }
        if (!list && tid < w.nw) {
            uint64_t m = 0;
            uint32_t c = 0;
            for (uint32_t q = 0; q < C; ++q) {
                m += *topo.map(&s.wmass[tid], q);
                c += *topo.map(&s.wcnt[tid], q);
            }
            s.wm_all[tid] = m;
            s.wc_all[tid] = c;
        }
        cta_sync();
        Z = s.b64[2];
        A = s.b64[3];
        CA = s.bu[7];
        tmass = (double)P * (double)Z;
        if (list) {
            const int n = gather_and_sort(topo, s);
            prefix_masses(s, r, n);
            if ((double)s.u.cd.pre[n] >= tmass) {  // the list holds the crossing
                nlist = n;
                break;
            }
        } else {
            uint64_t all = A;
            for (int g = 0; g < w.nw; ++g) all += s.wm_all[g];
            if ((double)A < tmass && (double)all >= tmass) break;
        }
    }

    if (nlist >= 0) {
        // list mode: the kept set is a prefix of the sorted list
        Crit cp;
        cp.by_mass = true;
        cp.tcnt = 1;
        cp.tmass = tmass;
        const Sel sp = walk_classes(s, nlist, cp, 0, 0);
        res.key_cut = sp.key;
        res.nk = sp.cnt;
        res.zk = sp.mass;
        const uint32_t kc = res.key_cut;
        for (int e = tid; e < (int)res.nk; e += kThreads) {  // kept entries of the list
            const uint64_t v = s.u.cd.sbuf[e];
            race.add(rc, dist(r, key_to_float(sb_key(v))), sb_idx(v));
        }
        res.token = race_finish(topo, s, src, r, rc, race.t2, kc);
        if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
        return res;
    }

    // the crossing group: the last group whose mass above is below tmass
    int gs = 0;
    uint64_t cum = A, C0 = CA, A0 = A;
    {
        uint64_t cnt = CA;
        for (int g = 0; g < w.nw; ++g) {
            if ((double)cum < tmass) {
                gs = g;
                A0 = cum;
                C0 = cnt;
            }
            cum += s.wm_all[g];
            cnt += s.wc_all[g];
        }
    }
    const int g_lo = w.b_lo + (gs << w.sh), g_end = min(w.b_lo + ((gs + 1) << w.sh), w.b_end);
    Crit cp;
    cp.by_mass = true;
    cp.tcnt = 1;
    cp.tmass = tmass;
    const Sel sp = refine_range(topo, s, src, r, zc, g_lo, g_end, key_k, cp, C0, A0);
    res.key_cut = max(sp.key, key_k);
    res.nk = sp.cnt;
    res.zk = sp.mass;
    // race over the window's kept tokens (those above the window were raced in the exact pass)
    const uint32_t kc = res.key_cut;
    const float flo = (float)w.b_lo;
    {
        RaceQueue<Src> rq(s);
        auto in_window = [&](float z) -> bool {  // kept, not raced yet, may race
            if (!((z > -INFINITY) && fkey(z) >= kc)) return false;
            const float d = dist(r, z);
            return !(d * kFineScale < flo) && !(16.64f - d < race.t2.k2);
        };
        src.for_each_vec(
            s,
            [&](const float* z, int v, bool ok) {
                uint32_t mask = 0;
                if (ok)
#pragma unroll
                    for (int j = 0; j < Src::kEPV; ++j)
                        if (in_window(z[j])) mask |= 1u << j;
                rq.push(src, r, rc, race, v, mask);
            },
            [&](float z, int32_t i) {
                if (in_window(z)) race.add(rc, dist(r, z), i);
            });
        rq.drain(src, r, rc, race);
    }
    res.token = race_finish(topo, s, src, r, rc, race.t2, kc);
    if (prow) write_probs(src, s, r, res.key_cut, res.zk, prow);
    return res;
}

// Per-row outputs (one thread of the writing CTA).  logprob: ln P(token); NaN for a failed row.
__device__ __forceinline__ void write_row(const Args& a, int64_t row, int32_t token, int32_t status, float cutoff,
                                          int32_t kept, float logprob)
{
    a.out_token[row] = token;
    if (a.out_status) a.out_status[row] = status;
    if (a.out_cutoff) a.out_cutoff[row] = cutoff;
    if (a.out_kept) a.out_kept[row] = kept;
    if (a.out_logprob) a.out_logprob[row] = logprob;
}
__device__ __forceinline__ void write_row(const Args& a, int64_t row, int32_t token, int32_t status, float cutoff,
                                          int32_t kept)
{
    write_row(a, row, token, status, cutoff, kept, __int_as_float(0x7FC00000));
}

// ln P(token) of a sampled row under the renormalised kept distribution: -(zmax - z)/T - ln(Z_kept)
// in double, the token's logit z read back from the row and Z_kept = zk 2^-44 (the exact fixed-point
// sum of the kept tokens' masses, relative to the maximum's).  Out of line: one call per row.
static __device__ __noinline__ float logprob_of(float zmax, float T, float z, uint64_t zk)
{
    const double dd = __ddiv_rn(__dsub_rn((double)zmax, (double)z), (double)T);
    return (float)(-dd - (log((double)zk) - 44.0 * 0.69314718055994530942));
}
// The general path sums the kept mass for a log-probability output even when no cut needs it.
__device__ __forceinline__ bool wants_zk(const Args& a) { return a.out_logprob != nullptr || a.out_top_idx != nullptr; }

template <typename TIn>
__device__ __forceinline__ float token_logprob(const Args& a, const RowCtx& r, int64_t row, int32_t token, uint64_t zk)
{
    if (!a.out_logprob) return 0.f;
    const float z = Elem<TIn>::load1(static_cast<const unsigned char*>(a.logits) + row * a.ld * Elem<TIn>::kBytes, token);
    return logprob_of(r.zmax, r.T, z, zk);
}

// The row's top tokens from its survivors sorted descending (key << 32 | ~index), the first nk of
// them kept: the most probable kept tokens with their ln P; slots past the kept ones get -1 and
// -inf.  Threads t, t + nthr, ... write slots t, t + nthr, ...
__device__ __forceinline__ void write_top(const Args& a, const RowCtx& r, int64_t row, const uint64_t* sorted,
                                          uint64_t nk, uint64_t zk, int t, int nthr)
{
    if (!a.out_top_idx) return;
    const int n = a.n_top;
    for (int j = t; j < n; j += nthr) {
        int32_t idx = -1;
        float lp = -INFINITY;
        if ((uint64_t)j < nk) {
            const uint64_t v = sorted[j];
            idx = sb_idx(v);
            lp = logprob_of(r.zmax, r.T, key_to_float(sb_key(v)), zk);
        }
        a.out_top_idx[row * n + j] = idx;
        a.out_top_logprob[row * n + j] = lp;
    }
}
// A greedy row: the token alone, ln P = 0.  A failed row: every slot -1 and NaN (token < 0).
__device__ __forceinline__ void write_top_single(const Args& a, int64_t row, int32_t token, int t, int nthr)
{
    if (!a.out_top_idx) return;
    const int n = a.n_top;
    for (int j = t; j < n; j += nthr) {
        const bool first = j == 0 && token >= 0;
        a.out_top_idx[row * n + j] = first ? token : -1;
        a.out_top_logprob[row * n + j] = first ? 0.f : (token >= 0 ? -INFINITY : __int_as_float(0x7FC00000));
    }
}

// The row's top kept tokens for the general path: the nk kept tokens are the top of the min-p
// survivors S0, so the first min(n_top, nk) of S0 in (logit desc, index asc) order are wanted.  The
// fine counts locate the bins that hold them; when those bins hold at most kCand survivors they are
// listed and sorted, otherwise the count cut is refined to the K-th largest logit first.  A tie
// class too large to list at that logit is resolved by extracting its lowest indices one pass at a
// time.  Every thread of every CTA of the topology calls it; `writer` threads write the outputs.
template <typename Topo, typename Src>
__device__ __noinline__ void general_top(Topo& topo, Shared& s, const Src& src, const RowCtx& r, float zc, uint64_t nk,
                           uint64_t zk, const Args& a, int64_t row, bool writer)
{
    if (!a.out_top_idx || a.n_top <= 0) return;
    cta_sync();  // the caller's block reductions are complete
    const uint64_t Kt = min((uint64_t)a.n_top, nk);
    const uint32_t* hr = topo.fine(s);
    int bn;
    uint64_t cn;
    fine_scan_topk(s, hr, Kt, &bn, &cn);
    uint32_t key_lo = 0;  // list the survivors with key >= key_lo inside bins <= bn
    if (cn + hr[bn] > (uint64_t)kCand) {
        Crit ck;
        ck.by_mass = false;
        ck.tcnt = Kt;
        ck.tmass = 0.0;
        const Sel sk = refine_range(topo, s, src, r, zc, bn, bn + 1, 0u, ck, cn, 0, false);
        key_lo = sk.key;
        if (sk.cnt > (uint64_t)kCand) key_lo = sk.key + 1u;  // the tie class at sk.key is resolved below
    }
    topo.sync();  // nobody still reads this CTA's lists or published values
    if (threadIdx.x == 0) s.ncand = 0;
    cta_sync();
    src.for_each(s, [&](float z, int32_t i) {
        if (!(z > zc)) return;
        const uint32_t key = fkey(z);
        if (key < key_lo) return;
        const float d = dist(r, z);
        if (fine_bin(d * kFineScale) > bn || !minp_ok(r, z, d)) return;
        const uint32_t slot = atomicAdd(&s.ncand, 1u);
        if (slot < (uint32_t)kCand) {
            s.ckey[slot] = key;
            s.cidx[slot] = (uint32_t)i;
        }
    });
    cta_sync();
    if (threadIdx.x == 0) s.pub_gcnt = min(s.ncand, (uint32_t)kCand);
    topo.sync();
    int n = gather_and_sort(topo, s);
    // A tie class too large to list: append its lowest indices, one pass each.
    if ((uint64_t)n < Kt && key_lo > 0) {
        const uint32_t tkey = key_lo - 1u;
        uint32_t last = 0;
        bool any = false;
        for (uint64_t j = (uint64_t)n; j < Kt; ++j) {
            uint32_t mi = 0xFFFFFFFFu;
            src.for_each(s, [&](float z, int32_t i) {
                if (z > -INFINITY && fkey(z) == tkey && (!any || (uint32_t)i > last)) mi = min(mi, (uint32_t)i);
            });
            mi = block_min_u32(mi, s);
            if (threadIdx.x == 0) s.pub_minidx = mi;
            topo.sync();
            if (threadIdx.x < 32) {
                uint32_t m = (threadIdx.x < topo.C) ? *topo.map(&s.pub_minidx, threadIdx.x) : 0xFFFFFFFFu;
                m = warp_min_u32(m);
                if (threadIdx.x == 0) s.bu[2] = m;
            }
            cta_sync();
            last = s.bu[2];
            any = true;
            if (threadIdx.x == 0) s.u.cd.sbuf[j] = sb_make(tkey, last);
            topo.sync();  // everyone has read pub_minidx
        }
        n = (int)Kt;
        cta_sync();
    }
    if (writer) write_top(a, r, row, s.u.cd.sbuf, min((uint64_t)n, Kt), zk, threadIdx.x, kThreads);
    cta_sync();
}

}  // namespace tps
