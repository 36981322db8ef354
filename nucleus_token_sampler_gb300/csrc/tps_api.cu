// tps_api.cu -- the C ABI declared in include/tps.h: argument checks, kernel and launch-shape
// choice, and the launches.  No host synchronisation, no state kept between calls beyond a
// per-device cache of queried limits.
//
// Two kernels sample the rows.  The cluster kernel (a thread-block cluster per row, the row held in
// the cluster's shared memory) spreads each row over up to 16 SMs; it samples small batches.  The
// streaming kernel (one persistent CTA per SM, rows streamed through a ring of bulk-copied chunks)
// reads each row once at HBM speed and resolves rows with min-p (and greedy rows) on the fly; its
// CTAs claim work dynamically through a small global scratch, which the call draws from a
// stream-ordered memory pool the library keeps per device and which a one-CTA kernel clears just
// before.  A large batch
// is split: the streaming kernel lists the rows without min-p (whose general path makes several
// passes over the row) in the scratch, and the cluster kernel, launched behind it, samples them.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "../../include/tps.h"
#include "tps_cluster.cuh"
#include "tps_kernels.h"
#include "tps_penalty.cuh"
#include "tps_reject.cuh"
#include "tps_spec.cuh"
#include "tps_stream.cuh"

namespace {

// The kernels for an element type (instantiated in their own translation units).
template <typename TIn>
tps::ClusterKernel cluster_kernel()
{
    return std::is_same<TIn, float>::value ? tps::cluster_kernel_f32() : tps::cluster_kernel_bf16();
}
template <typename TIn>
tps::StreamKernel stream_kernel()
{
    return std::is_same<TIn, float>::value ? tps::stream_kernel_f32() : tps::stream_kernel_bf16();
}

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxVocabMass = (int64_t(1) << 20) - 1;  // fixed-point mass sums fit 64 bits
constexpr uint32_t kSliceTarget = 64u * 1024u;              // preferred slice per CTA
constexpr int kMaxCluster = 16;

constexpr int kStreamStages = 3;
constexpr uint32_t kStreamChunk = 64u * 1024u;
constexpr int64_t kStreamMinRows = 32;  // batches at least this large use the streaming kernel
constexpr int64_t kMinSegBytes = 128 * 1024;  // smallest segment of a split row
constexpr int kClaimsPerSm = 4;                // claims per SM below which rows are split

// Per-device limits, filled once under g_mu and published through `ready` (release/acquire), so a
// thread that sees ready == true also sees sms and smem_optin.  The attribute flags only record that
// cudaFuncSetAttribute has succeeded once; setting an attribute twice is harmless, so they need no
// lock, only atomic access.
struct DeviceInfo {
    std::atomic<bool> ready{false};
    int sms = 0;
    int smem_optin = 0;
    std::atomic<bool> attrs_f32{false}, attrs_bf16{false};
    std::atomic<bool> sattrs_f32{false}, sattrs_bf16{false};
    // Largest dynamic shared memory per CTA seen to co-schedule a cluster of 9..16 CTAs, per dtype
    // (0 = not known yet).
    std::atomic<long> wide_ok[2][kMaxCluster + 1];
    // Co-resident clusters per (dtype, cluster size): shared-memory bytes << 20 | count (0 = not known).
    std::atomic<long> resident[2][kMaxCluster + 1];
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

// The library's own stream-ordered memory pool per device, for the streaming kernel's per-call
// scratch.  The device's default pool gives all unused memory back at every synchronisation, so the
// first call after a cudaStreamSynchronize would map fresh memory on the host's critical path; this
// pool keeps up to kPoolKeepBytes reserved instead (a call's scratch is a few KB for a batch of whole
// rows and at most about 2.5 MB for a split batch).  Created once per device, with that device current, and kept until the
// process exits.
constexpr uint64_t kPoolKeepBytes = 64ull << 20;
std::atomic<cudaMemPool_t> g_pool[kMaxDevices];
std::mutex g_pool_mu;

cudaError_t scratch_pool(cudaMemPool_t* out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaMemPool_t p = g_pool[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        p = g_pool[dev].load(std::memory_order_relaxed);
        if (!p) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            e = cudaMemPoolCreate(&p, &props);
            if (e != cudaSuccess) return e;
            uint64_t keep = kPoolKeepBytes;
            e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
            if (e != cudaSuccess) {
                cudaMemPoolDestroy(p);
                return e;
            }
            g_pool[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return cudaSuccess;
}

int elem_bytes(int dtype) { return dtype == TPS_F32 ? 4 : (dtype == TPS_BF16 ? 2 : 0); }

bool device_info(DeviceInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0, optin = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
            if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
                return false;
            d.sms = sms;
            d.smem_optin = optin;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return true;
}

// Slice bytes a CTA must hold for a row of V elements split over C CTAs (upper bound over every
// alignment of the row start), rounded to 128 bytes.
uint32_t slice_cap_bytes(int64_t V, int es, int C)
{
    const int64_t n16 = (V * es) / 16;          // aligned interior vectors, at most
    const int64_t per = (n16 + C - 1) / C;      // per CTA
    return (uint32_t)(((per * 16) + 127) / 128 * 128);
}

// Slice, shared state, the cluster-wide fine histogram, a spare row list and the exchange inbox.
size_t smem_bytes(uint32_t slice_cap)
{
    return (size_t)slice_cap + sizeof(tps::Shared) + 2 * (size_t)tps::kFineBins * sizeof(uint32_t) +
           (size_t)tps::kThreads * sizeof(int32_t) + sizeof(tps::Inbox);
}

// The streaming kernel's work for B rows: rows [0, b_whole) are claimed whole, the last nsplit rows
// as nseg segments each.  A batch of at least kClaimsPerSm rows per SM is streamed in whole rows:
// claims are dynamic, so the SMs finish within about one row of each other, and a split row costs a
// merge of its segments' partial results through the scratch at the end of the row.  A smaller batch
// would leave SMs idle, so every row is split into enough segments (of at least kMinSegBytes, at most
// tps::kMaxSegments) to give about kClaimsPerSm claims per SM.
struct StreamPlan {
    int64_t b_whole, nsplit;
    int nseg;
    int64_t claims;
    int grid;
    tps::ScratchLayout layout;
};
StreamPlan stream_plan(const DeviceInfo& d, int64_t B, int64_t V, int es)
{
    StreamPlan p;
    const int64_t row_bytes = V * es;
    const int64_t want = kClaimsPerSm * (int64_t)d.sms;
    int64_t nseg = 1;
    if (B < want)
        nseg = std::min<int64_t>(std::min<int64_t>((want + B - 1) / B, row_bytes / kMinSegBytes), tps::kMaxSegments);
    p.nseg = (int)std::max<int64_t>(1, nseg);
    p.nsplit = p.nseg > 1 ? B : 0;
    p.b_whole = B - p.nsplit;
    p.claims = p.b_whole + p.nsplit * p.nseg;
    p.grid = (int)std::min<int64_t>(d.sms, p.claims);
    p.layout = tps::ScratchLayout::of(B, p.nsplit, p.nseg);
    return p;
}

// Zero the part of a streaming call's scratch that must start at zero (counters), then let the
// streaming kernel, launched behind this one as its programmatic dependent, start at once: it
// reads logits and parameters right away and waits for this grid only before its first claim.
__global__ void clear_scratch_kernel(uint32_t* p, uint32_t nwords)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (uint32_t i = threadIdx.x; i < nwords; i += blockDim.x) p[i] = 0u;
}

// Choose the cluster size: the smallest C whose slice fits the preferred size, widened for small
// batches so one row spreads over more SMs.  Returns 0 if even 16 CTAs cannot hold the row.
int choose_cluster(const DeviceInfo& d, int es, int64_t B, int64_t V)
{
    const int64_t row_bytes = V * es;
    int c = (int)((row_bytes + kSliceTarget - 1) / kSliceTarget);
    if (c < 1) c = 1;
    if (B > 0 && B * 2 <= d.sms) {
        int want = (int)(d.sms / B);
        if (want > kMaxCluster) want = kMaxCluster;
        if (want > c) c = want;
    }
    if (V < 64 * (int64_t)c) {  // tiny rows: do not spread a handful of vectors over many CTAs
        c = (int)((V + 63) / 64);
        if (c < 1) c = 1;
    }
    while (c <= kMaxCluster && smem_bytes(slice_cap_bytes(V, es, c)) > (size_t)d.smem_optin) ++c;
    if (c > kMaxCluster) return 0;
    return c;
}

template <typename TIn>
cudaError_t prepare_kernel(const DeviceInfo& d)
{
    auto k = cluster_kernel<TIn>();
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem_optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

// Clusters of more than 8 CTAs are not guaranteed to fit a GPC; ask the occupancy calculator
// once per (dtype, cluster size, shared-memory size) and fall back to 8 when they do not.
template <typename TIn>
bool wide_cluster_ok(DeviceInfo& d, int dt, int C, size_t smem)
{
    std::atomic<long>& slot = d.wide_ok[dt][C];
    const long known = slot.load();
    if (known > 0 && (size_t)known >= smem) return true;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(tps::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, cluster_kernel<TIn>(), &cfg);
    if (e != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        return false;
    }
    if ((long)smem > known) slot.store((long)smem);
    return true;
}

constexpr size_t kSmemPerBlockMax = 232448;  // 227 KB opt-in shared memory per CTA on sm_100/sm_103
static_assert((size_t)kStreamStages * kStreamChunk + sizeof(tps::Shared) + sizeof(tps::StreamState) <= kSmemPerBlockMax,
              "the streaming kernel's ring and state must fit one CTA's shared memory");

static_assert(tps::kMaxHistory == TPS_MAX_HISTORY && 2 * tps::penalty_slots(TPS_MAX_HISTORY) * sizeof(uint32_t) <= kSmemPerBlockMax,
              "the penalty kernel's hash table for the longest history fits one CTA's shared memory");

size_t stream_smem_bytes() { return (size_t)kStreamStages * kStreamChunk + sizeof(tps::Shared) + sizeof(tps::StreamState); }

// The streaming kernel over `grid` CTAs, as the programmatic dependent of the clear kernel
// launched just before it.
template <typename TIn>
cudaError_t launch_stream(std::atomic<bool>* attrs_done, const tps::Args& a, int grid, cudaStream_t stream)
{
    auto k = stream_kernel<TIn>();
    const size_t smem = stream_smem_bytes();
    if (!attrs_done->load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attrs_done->store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(tps::kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a, (int)kStreamStages, (uint32_t)kStreamChunk);
}

// The cluster kernel over `nclusters` clusters of C CTAs; `dependent`: as the programmatic
// dependent of the streaming kernel launched just before it (list mode).
template <typename TIn>
cudaError_t launch(const tps::Args& a, int C, size_t smem, int64_t nclusters, bool dependent, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nclusters * C), 1, 1);
    cfg.blockDim = dim3(tps::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, cluster_kernel<TIn>(), a);
}

// Clusters of C CTAs the device holds at once (at least 1), asked once per (dtype, C, shared memory).
template <typename TIn>
int64_t resident_clusters(DeviceInfo& d, int dt, int C, size_t smem)
{
    std::atomic<long>& slot = d.resident[dt][C];
    const long known = slot.load();
    if (known > 0 && (size_t)(known >> 20) == smem) return known & 0xFFFFF;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(tps::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, cluster_kernel<TIn>(), &cfg) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    if (n > 0xFFFFF) n = 0xFFFFF;
    slot.store(((long)smem << 20) | (long)n);
    return n;
}

int fail_cuda(cudaError_t e)
{
    g_last_cuda_error = (int)e;
    return TPS_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


// One sampling call's arguments (the C ABI's, gathered).
struct Call {
    const void* logits;
    int dtype;
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
    float* out_logprob;
    int32_t n_top;
    int32_t* out_top_idx;
    float* out_top_logprob;
    int kernel;
    cudaStream_t stream;
    uint64_t wait_ns = tps::kWaitLimitNs;
    int64_t stall_chunk = -1;
};

// Where a streaming call's scratch comes from: the library's stream-ordered pool, or a fixed array
// (`fixed`, `fixed_bytes`) the call uses as it is.
enum class ScratchSource { kPool, kFixed };

int sample_call(const Call& c, ScratchSource src, void* fixed = nullptr, size_t fixed_bytes = 0)
{
    const int64_t B = c.B, V = c.V;
    if (c.kernel < TPS_KERNEL_AUTO || c.kernel > TPS_KERNEL_STREAM) return TPS_ERR_ARG;
    if (B < 0 || V < 1 || c.ld < V || c.n_top < 0 || c.n_top > TPS_MAX_TOP) return TPS_ERR_ARG;
    if (c.n_top > 0 && (!c.out_top_idx || !c.out_top_logprob)) return TPS_ERR_ARG;
    const int es = elem_bytes(c.dtype);
    if (!es) return TPS_ERR_DTYPE;
    if (B == 0) return TPS_OK;
    if (!c.logits || !c.temperature || !c.top_k || !c.top_p || !c.min_p || !c.seed || !c.out_token) return TPS_ERR_ARG;
    if (!aligned(c.logits, es) || !aligned(c.temperature, 4) || !aligned(c.top_k, 4) || !aligned(c.top_p, 4) ||
        !aligned(c.min_p, 4) || !aligned(c.seed, 8) || !aligned(c.out_token, 4) ||
        (c.out_probs && !aligned(c.out_probs, 4)) || (c.out_status && !aligned(c.out_status, 4)) ||
        (c.out_cutoff && !aligned(c.out_cutoff, 4)) || (c.out_kept && !aligned(c.out_kept, 4)) ||
        (c.out_logprob && !aligned(c.out_logprob, 4)) ||
        (c.n_top > 0 && (!aligned(c.out_top_idx, 4) || !aligned(c.out_top_logprob, 4))))
        return TPS_ERR_ALIGN;
    if (V > kMaxVocabMass || V > INT32_MAX) return TPS_ERR_UNSUPPORTED_V;
    if (B > (int64_t)INT32_MAX / kMaxCluster) return TPS_ERR_ARG;

    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return fail_cuda(cudaGetLastError());
    const int Cfit = choose_cluster(*d, es, B, V);
    const int kernel = c.kernel;
    const bool use_stream = kernel == TPS_KERNEL_STREAM || (kernel == TPS_KERNEL_AUTO && B >= kStreamMinRows) ||
                            (kernel == TPS_KERNEL_AUTO && Cfit == 0);
    // A large batch is split: the streaming kernel takes the rows with min-p (and greedy and failed
    // rows) and lists the others, which the cluster kernel, launched behind it, samples.
    const bool split = kernel == TPS_KERNEL_AUTO && use_stream && Cfit != 0;
    if (!use_stream && Cfit == 0) return TPS_ERR_UNSUPPORTED_V;

    tps::Args a = {};
    a.logits = c.logits;
    a.B = B;
    a.V = V;
    a.ld = c.ld;
    a.temperature = c.temperature;
    a.top_k = c.top_k;
    a.top_p = c.top_p;
    a.min_p = c.min_p;
    a.seed = c.seed;
    a.step = c.step;
    a.out_token = c.out_token;
    a.out_probs = c.out_probs;
    a.out_status = c.out_status;
    a.out_cutoff = c.out_cutoff;
    a.out_kept = c.out_kept;
    a.out_logprob = c.out_logprob;
    a.n_top = c.n_top;
    a.out_top_idx = c.n_top > 0 ? c.out_top_idx : nullptr;
    a.out_top_logprob = c.n_top > 0 ? c.out_top_logprob : nullptr;
    a.wait_ns = c.wait_ns;
    a.stall_chunk = c.stall_chunk;
    const cudaStream_t st = c.stream;
    cudaError_t e;

    // The cluster kernel's shape (for a cluster-only call, or the list mode of a split batch).
    int Cl = Cfit;
    uint32_t cap = Cfit ? slice_cap_bytes(V, es, Cfit) : 0u;
    size_t sm = smem_bytes(cap);
    if (!use_stream || split) {
        const int dt = c.dtype == TPS_F32 ? 0 : 1;
        std::atomic<bool>& done = c.dtype == TPS_F32 ? d->attrs_f32 : d->attrs_bf16;
        if (!done.load(std::memory_order_acquire)) {
            e = c.dtype == TPS_F32 ? prepare_kernel<float>(*d) : prepare_kernel<__nv_bfloat16>(*d);
            if (e != cudaSuccess) return fail_cuda(e);
            done.store(true, std::memory_order_release);
        }
        // a cluster wider than 8 that the GPU cannot co-schedule falls back to 8 CTAs, if they hold the row
        if (Cl > 8) {
            const bool wide = c.dtype == TPS_F32 ? wide_cluster_ok<float>(*d, dt, Cl, sm)
                                                 : wide_cluster_ok<__nv_bfloat16>(*d, dt, Cl, sm);
            if (!wide) {
                if (smem_bytes(slice_cap_bytes(V, es, 8)) > (size_t)d->smem_optin) return TPS_ERR_UNSUPPORTED_V;
                Cl = 8;
                cap = slice_cap_bytes(V, es, 8);
                sm = smem_bytes(cap);
            }
        }
    }
    if (!use_stream) {  // the cluster kernel alone, one cluster per row
        a.route = tps::kRouteAll;
        a.slice_cap = cap;
        e = c.dtype == TPS_F32 ? launch<float>(a, Cl, sm, B, false, st) : launch<__nv_bfloat16>(a, Cl, sm, B, false, st);
        return e == cudaSuccess ? TPS_OK : fail_cuda(e);
    }

    // The streaming kernel (and, for a split batch, the cluster kernel behind it) with its scratch.
    const StreamPlan pl = stream_plan(*d, B, V, es);
    void* scratch = nullptr;
    if (src == ScratchSource::kPool) {
        cudaMemPool_t pool = nullptr;
        e = scratch_pool(&pool);
        if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&scratch, (size_t)pl.layout.total, pool, st);
        if (e != cudaSuccess) return fail_cuda(e);
    } else {
        if (pl.layout.total > (uint64_t)fixed_bytes) return TPS_ERR_SCRATCH;
        scratch = fixed;
    }
    a.scratch = scratch;
    a.b_whole = pl.b_whole;
    a.nsplit = pl.nsplit;
    a.nseg = pl.nseg;
    a.route = split ? tps::kRouteStream : tps::kRouteAll;
    a.slice_cap = 0;
    clear_scratch_kernel<<<1, 256, 0, st>>>(static_cast<uint32_t*>(scratch), (uint32_t)(pl.layout.clear_bytes() / 4));
    e = cudaGetLastError();
    if (e == cudaSuccess)
        e = c.dtype == TPS_F32 ? launch_stream<float>(&d->sattrs_f32, a, pl.grid, st)
                               : launch_stream<__nv_bfloat16>(&d->sattrs_bf16, a, pl.grid, st);
    if (e == cudaSuccess && split) {
        a.route = tps::kRouteList;
        a.slice_cap = cap;
        const int dt = c.dtype == TPS_F32 ? 0 : 1;
        const int64_t ncl = std::min<int64_t>(B, c.dtype == TPS_F32 ? resident_clusters<float>(*d, dt, Cl, sm)
                                                                    : resident_clusters<__nv_bfloat16>(*d, dt, Cl, sm));
        e = c.dtype == TPS_F32 ? launch<float>(a, Cl, sm, ncl, true, st) : launch<__nv_bfloat16>(a, Cl, sm, ncl, true, st);
    }
    if (src == ScratchSource::kPool) {
        const cudaError_t ef = cudaFreeAsync(scratch, st);
        if (e == cudaSuccess) e = ef;
    }
    return e == cudaSuccess ? TPS_OK : fail_cuda(e);
}

}  // namespace

extern "C" {

int tps_version(void) { return 100; }

int tps_last_cuda_error(void) { return g_last_cuda_error; }

const char* tps_status_string(int status)
{
    switch (status) {
    case TPS_OK: return "ok";
    case TPS_ERR_ARG: return "invalid argument (null pointer, B < 0, V < 1 or ld < V)";
    case TPS_ERR_DTYPE: return "unknown dtype";
    case TPS_ERR_UNSUPPORTED_V: return "vocabulary too large for this device";
    case TPS_ERR_ALIGN: return "pointer not aligned to its element type";
    case TPS_ERR_CUDA: return "CUDA runtime error";
    case TPS_ERR_SCRATCH: return "the call needs more scratch than the fixed scratch array of tps_sample_noalloc holds";
    case 100 + TPS_ROW_OK: return "row ok";
    case 100 + TPS_ROW_NAN: return "row holds a NaN or +inf logit";
    case 100 + TPS_ROW_ALL_MASKED: return "every logit of the row is -inf";
    case 100 + TPS_ROW_BAD_PARAM: return "temperature, top_p or min_p is not finite";
    case 100 + TPS_ROW_TIMEOUT: return "a bounded wait in the kernel gave up";
    default: return "unknown status";
    }
}

int64_t tps_max_vocab(int dtype)
{
    // The streaming kernel holds no row in shared memory; the limit is the exact 64-bit mass sum.
    const int es = elem_bytes(dtype);
    if (!es) return 0;
    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return 0;
    return kMaxVocabMass;
}

int tps_kernels_per_call(int dtype, int64_t B, int64_t V, int kernel)
{
    const int es = elem_bytes(dtype);
    if (!es || V < 1 || B < 0 || V > kMaxVocabMass || kernel < TPS_KERNEL_AUTO || kernel > TPS_KERNEL_STREAM) return 0;
    if (B == 0) return 0;
    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return 0;
    const int Cfit = choose_cluster(*d, es, B, V);
    if (kernel == TPS_KERNEL_CLUSTER) return Cfit ? 1 : 0;
    if (kernel == TPS_KERNEL_STREAM) return 2;  // the scratch clear, the streaming kernel
    if (B < kStreamMinRows && Cfit != 0) return 1;
    return Cfit != 0 ? 3 : 2;  // auto: a large batch is split (clear, streaming, cluster)
}

int tps_cluster_size(int dtype, int64_t B, int64_t V)
{
    const int es = elem_bytes(dtype);
    if (!es || V < 1 || B < 0) return 0;
    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return 0;
    if (V > kMaxVocabMass) return 0;
    return choose_cluster(*d, es, B, V);
}

int tps_sample_full(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                    const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                    uint64_t step, int32_t* out_token, float* out_probs, int32_t* out_status, float* out_cutoff,
                    int32_t* out_kept, float* out_logprob, int32_t n_top, int32_t* out_top_idx,
                    float* out_top_logprob, int kernel, void* stream)
{
    Call c;
    c.logits = logits;
    c.dtype = dtype;
    c.B = B;
    c.V = V;
    c.ld = ld;
    c.temperature = temperature;
    c.top_k = top_k;
    c.top_p = top_p;
    c.min_p = min_p;
    c.seed = seed;
    c.step = step;
    c.out_token = out_token;
    c.out_probs = out_probs;
    c.out_status = out_status;
    c.out_cutoff = out_cutoff;
    c.out_kept = out_kept;
    c.out_logprob = out_logprob;
    c.n_top = n_top;
    c.out_top_idx = out_top_idx;
    c.out_top_logprob = out_top_logprob;
    c.kernel = kernel;
    c.stream = static_cast<cudaStream_t>(stream);
    return sample_call(c, ScratchSource::kPool);
}

int tps_apply_penalties(void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const int32_t* history, int64_t H,
                        int64_t ldh, const int32_t* hist_len, const float* repetition, const float* frequency,
                        const float* presence, int32_t* out_status, void* stream)
{
    if (B < 0 || V < 1 || ld < V || H < 0 || H > TPS_MAX_HISTORY || ldh < H) return TPS_ERR_ARG;
    const int es = elem_bytes(dtype);
    if (!es) return TPS_ERR_DTYPE;
    if (B == 0) return TPS_OK;
    if (!logits || (H > 0 && !history)) return TPS_ERR_ARG;
    if (!aligned(logits, es) || (history && !aligned(history, 4)) || (hist_len && !aligned(hist_len, 4)) ||
        (repetition && !aligned(repetition, 4)) || (frequency && !aligned(frequency, 4)) ||
        (presence && !aligned(presence, 4)) || (out_status && !aligned(out_status, 4)))
        return TPS_ERR_ALIGN;
    if (V > INT32_MAX) return TPS_ERR_UNSUPPORTED_V;
    if (!repetition && !frequency && !presence && !out_status) return TPS_OK;  // nothing to change or report

    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return fail_cuda(cudaGetLastError());
    tps::PenaltyArgs a;
    a.logits = logits;
    a.B = B;
    a.V = V;
    a.ld = ld;
    a.hist = history;
    a.H = H;
    a.ldh = ldh;
    a.hist_len = hist_len;
    a.rep = repetition;
    a.freq = frequency;
    a.pres = presence;
    a.out_status = out_status;
    const cudaError_t e = tps::launch_penalties(a, dtype == TPS_BF16, d->sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    return TPS_OK;
}

int tps_sample_stall_test(const void* logits, int dtype, int64_t B, int64_t V, const float* temperature,
                          const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                          uint64_t step, int32_t* out_token, int32_t* out_status, int64_t stall_chunk,
                          uint64_t wait_ns, void* stream)
{
    if (wait_ns == 0 || wait_ns > tps::kWaitLimitNs) return TPS_ERR_ARG;
    Call c;
    c.logits = logits;
    c.dtype = dtype;
    c.B = B;
    c.V = V;
    c.ld = V;
    c.temperature = temperature;
    c.top_k = top_k;
    c.top_p = top_p;
    c.min_p = min_p;
    c.seed = seed;
    c.step = step;
    c.out_token = out_token;
    c.out_probs = nullptr;
    c.out_status = out_status;
    c.out_cutoff = nullptr;
    c.out_kept = nullptr;
    c.out_logprob = nullptr;
    c.n_top = 0;
    c.out_top_idx = nullptr;
    c.out_top_logprob = nullptr;
    c.kernel = TPS_KERNEL_STREAM;
    c.stream = static_cast<cudaStream_t>(stream);
    c.wait_ns = wait_ns;
    c.stall_chunk = stall_chunk;
    return sample_call(c, ScratchSource::kPool);
}

int tps_sample_rejection(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                         const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                         uint64_t step, int32_t* out_token, int32_t* out_status, float* out_cutoff, int32_t* out_kept,
                         int32_t* out_rounds, void* stream)
{
    if (B < 0 || V < 1 || ld < V) return TPS_ERR_ARG;
    const int es = elem_bytes(dtype);
    if (!es) return TPS_ERR_DTYPE;
    if (B == 0) return TPS_OK;
    if (!logits || !temperature || !top_k || !top_p || !min_p || !seed || !out_token) return TPS_ERR_ARG;
    if (!aligned(logits, es) || !aligned(temperature, 4) || !aligned(top_k, 4) || !aligned(top_p, 4) ||
        !aligned(min_p, 4) || !aligned(seed, 8) || !aligned(out_token, 4) || (out_status && !aligned(out_status, 4)) ||
        (out_cutoff && !aligned(out_cutoff, 4)) || (out_kept && !aligned(out_kept, 4)) ||
        (out_rounds && !aligned(out_rounds, 4)))
        return TPS_ERR_ALIGN;
    if (V > kMaxVocabMass || V > INT32_MAX) return TPS_ERR_UNSUPPORTED_V;
    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return fail_cuda(cudaGetLastError());
    tps::RejectArgs ra = {};
    ra.a.logits = logits;
    ra.a.B = B;
    ra.a.V = V;
    ra.a.ld = ld;
    ra.a.temperature = temperature;
    ra.a.top_k = top_k;
    ra.a.top_p = top_p;
    ra.a.min_p = min_p;
    ra.a.seed = seed;
    ra.a.step = step;
    ra.a.out_token = out_token;
    ra.a.out_status = out_status;
    ra.a.out_cutoff = out_cutoff;
    ra.a.out_kept = out_kept;
    ra.out_rounds = out_rounds;
    const cudaError_t e = tps::launch_reject(ra, dtype == TPS_BF16, d->sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TPS_OK : fail_cuda(e);
}

int tps_spec_accept(const void* target_logits, const void* draft_logits, int dtype, int64_t B, int64_t V, int64_t ld,
                    const float* target_temperature, const int32_t* target_top_k, const float* target_top_p,
                    const float* target_min_p, const float* draft_temperature, const int32_t* draft_top_k,
                    const float* draft_top_p, const float* draft_min_p, const int32_t* draft_token,
                    const uint64_t* seed, uint64_t step, int32_t* out_token, int32_t* out_accepted,
                    int32_t* out_status, void* stream)
{
    if (B < 0 || V < 1 || ld < V) return TPS_ERR_ARG;
    const int es = elem_bytes(dtype);
    if (!es) return TPS_ERR_DTYPE;
    if (B == 0) return TPS_OK;
    if (!target_logits || !draft_logits || !target_temperature || !target_top_k || !target_top_p || !target_min_p ||
        !draft_temperature || !draft_top_k || !draft_top_p || !draft_min_p || !draft_token || !seed || !out_token)
        return TPS_ERR_ARG;
    if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(target_temperature, 4) ||
        !aligned(target_top_k, 4) || !aligned(target_top_p, 4) || !aligned(target_min_p, 4) ||
        !aligned(draft_temperature, 4) || !aligned(draft_top_k, 4) || !aligned(draft_top_p, 4) ||
        !aligned(draft_min_p, 4) || !aligned(draft_token, 4) || !aligned(seed, 8) || !aligned(out_token, 4) ||
        (out_accepted && !aligned(out_accepted, 4)) || (out_status && !aligned(out_status, 4)))
        return TPS_ERR_ALIGN;
    if (V > kMaxVocabMass || V > INT32_MAX) return TPS_ERR_UNSUPPORTED_V;
    DeviceInfo* d = nullptr;
    if (!device_info(&d)) return fail_cuda(cudaGetLastError());
    tps::SpecArgs a;
    a.target = target_logits;
    a.draft = draft_logits;
    a.B = B;
    a.V = V;
    a.ld = ld;
    a.tT = target_temperature;
    a.tK = target_top_k;
    a.tP = target_top_p;
    a.tM = target_min_p;
    a.dT = draft_temperature;
    a.dK = draft_top_k;
    a.dP = draft_top_p;
    a.dM = draft_min_p;
    a.draft_token = draft_token;
    a.seed = seed;
    a.step = step;
    a.out_token = out_token;
    a.out_accepted = out_accepted;
    a.out_status = out_status;
    const cudaError_t e = tps::launch_spec(a, dtype == TPS_BF16, d->sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TPS_OK : fail_cuda(e);
}

int tps_sample_kernel(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                      const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                      uint64_t step, int32_t* out_token, float* out_probs, int32_t* out_status, float* out_cutoff,
                      int32_t* out_kept, int kernel, void* stream)
{
    return tps_sample_full(logits, dtype, B, V, ld, temperature, top_k, top_p, min_p, seed, step, out_token, out_probs,
                           out_status, out_cutoff, out_kept, nullptr, 0, nullptr, nullptr, kernel, stream);
}

int tps_sample_ex(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                  const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed, uint64_t step,
                  int32_t* out_token, float* out_probs, int32_t* out_status, float* out_cutoff, int32_t* out_kept,
                  void* stream)
{
    return tps_sample_kernel(logits, dtype, B, V, ld, temperature, top_k, top_p, min_p, seed, step, out_token,
                             out_probs, out_status, out_cutoff, out_kept, TPS_KERNEL_AUTO, stream);
}

int tps_sample(const void* logits, int dtype, int64_t B, int64_t V, const float* temperature, const int32_t* top_k,
               const float* top_p, const float* min_p, const uint64_t* seed, uint64_t step, int32_t* out_token,
               float* out_probs, void* stream)
{
    return tps_sample_ex(logits, dtype, B, V, V, temperature, top_k, top_p, min_p, seed, step, out_token,
                         out_probs, nullptr, nullptr, nullptr, stream);
}

}  // extern "C"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocAddr {
    std::atomic<bool> ready{false};
    void* ptr = nullptr;
};
NoAllocAddr g_noalloc_addr[kMaxDevices];
std::mutex g_noalloc_mu;

// The fixed array's device address on the current device (looked up once per device).
cudaError_t noalloc_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    NoAllocAddr& na = g_noalloc_addr[dev];
    if (!na.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!na.ready.load(std::memory_order_relaxed)) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            na.ptr = p;
            na.ready.store(true, std::memory_order_release);
        }
    }
    *out = na.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------------------------
// tps_sample_noalloc: the sampling call for callers that cannot allocate device memory.  Some
// callers may not allocate on the device at all while they sample: a serving loop that reserves
// all device memory up front and must not meet an allocation failure mid-request, a host whose
// allocator is owned by another framework (allocating behind its back would break its accounting),
// or code that must not enter the driver's allocator for latency reasons.  The ordinary calls draw
// the streaming kernel's small per-call scratch from the library's stream-ordered pool
// (cudaMallocFromPoolAsync); this call uses a fixed array compiled into the library instead.  The array is
// kNoAllocScratchBytes of device memory on every GPU that loads the library, held until the process
// exits.  Its device address is looked up once per device (cudaGetSymbolAddress, with that device
// current) by the first call on that device, so that first call should come before any stream
// capture.  Every call shares the one array and leaves its last contents there: the part that must
// start at zero (the claim and arrival counters) is cleared by each call's own clearing kernel, on the
// call's stream.  Two calls that overlap on the GPU (different streams, no ordering between them)
// race on the array and must not be issued.
// ---------------------------------------------------------------------------------------------
int tps_sample_noalloc(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                       const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                       uint64_t step, int32_t* out_token, float* out_probs, int32_t* out_status, float* out_cutoff,
                       int32_t* out_kept, float* out_logprob, int32_t n_top, int32_t* out_top_idx,
                       float* out_top_logprob, int kernel, void* stream)
{
    Call c;
    c.logits = logits;
    c.dtype = dtype;
    c.B = B;
    c.V = V;
    c.ld = ld;
    c.temperature = temperature;
    c.top_k = top_k;
    c.top_p = top_p;
    c.min_p = min_p;
    c.seed = seed;
    c.step = step;
    c.out_token = out_token;
    c.out_probs = out_probs;
    c.out_status = out_status;
    c.out_cutoff = out_cutoff;
    c.out_kept = out_kept;
    c.out_logprob = out_logprob;
    c.n_top = n_top;
    c.out_top_idx = out_top_idx;
    c.out_top_logprob = out_top_logprob;
    c.kernel = kernel;
    c.stream = static_cast<cudaStream_t>(stream);
    void* scratch = nullptr;
    const cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    return sample_call(c, ScratchSource::kFixed, scratch, kNoAllocScratchBytes);
}

}  // extern "C"
