// tps_penalty.cuh -- repetition, frequency and presence penalties on the raw logits, the stage a
// serving engine runs ahead of the sampler ("Top-p (Nucleus) Sampling, in depth", "Where top-p
// sits in the sampler chain": penalties come first, on the logits; "What do temperature, top-k and
// top-p each do ...", "What interviewers probe next": before temperature, on raw logits, so they
// move the greedy choice too).  The pages give no formulas; the kernel applies the common ones to
// every token t that occurs c_t > 0 times in the row's history:
//     y = z_t / r  if z_t > 0,  z_t * r otherwise;     z'_t = y - (f * c_t + rho)
// in float32, one correctly rounded operation at a time (no contraction), rounded to nearest-even
// bfloat16 for bfloat16 logits.  Every other logit is left as it is.
//
// One CTA of 512 threads per row (up to 64 CTAs per SM, grid-stride beyond).  The row's valid
// history ids (those in [0, V)) are counted in a shared-memory hash table of at least twice the
// history length (open addressing, linear probing; the lanes of a warp holding the same id are
// grouped with a match, and the group's leader claims the slot with a compare-and-swap and adds
// the group's size); then every occupied slot rewrites its token with the count.  Each token is
// written by one thread with its exact count whatever the slot layout, so the result is
// deterministic; three barriers per row.  History entries and the logits a thread rewrites are
// loaded four at a time, so their latencies overlap.  Memory traffic per row: the history (4 B per
// entry) plus a read and a write of each distinct token's logit.
#pragma once

#include "tps_common.cuh"

namespace tps {

constexpr int kPenaltyThreads = 512;
constexpr int kMaxHistory = 8192;  // history entries per row (a 128 KB hash table)

struct PenaltyArgs {
    void* logits;             // [B, ld], modified in place
    int64_t B, V, ld;
    const int32_t* hist;      // [B, ldh] token ids
    int64_t H, ldh;
    const int32_t* hist_len;  // [B] or null (every row uses H)
    const float* rep;         // [B] or null (1)
    const float* freq;        // [B] or null (0)
    const float* pres;        // [B] or null (0)
    int32_t* out_status;      // [B] or null
};

__device__ __forceinline__ float pen_load(const float* p) { return *p; }
__device__ __forceinline__ float pen_load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void pen_store(float* p, float v) { *p = v; }
__device__ __forceinline__ void pen_store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

constexpr int kBatch = 4;  // history entries / table slots a thread handles per round

// Count `k` occurrences of id t in the table (open addressing, linear probing).  At most n <= S/2
// distinct ids are inserted, so a slot is always found within S probes.
__device__ __forceinline__ void count_id(uint32_t* keys, uint32_t* cnt, uint32_t t, uint32_t k, int S, int sh)
{
    uint32_t s = (t * 0x9E3779B1u) >> sh;
    for (int probe = 0; probe < S; ++probe) {
        const uint32_t prev = atomicCAS(&keys[s], 0xFFFFFFFFu, t);
        if (prev == 0xFFFFFFFFu || prev == t) {
            atomicAdd(&cnt[s], k);
            return;
        }
        s = (s + 1u) & (uint32_t)(S - 1);
    }
}

// Hash-table slots for a history of n entries: a power of two >= max(2 n, 64).
__host__ __device__ constexpr int penalty_slots(int64_t n)
{
    int S = 64;
    while (S < 2 * n) S <<= 1;
    return S;
}

template <typename TIn>
__global__ void __launch_bounds__(kPenaltyThreads, 4) penalty_rows_kernel(const PenaltyArgs a)
{
    extern __shared__ uint32_t sm[];  // keys[S], counts[S] with S = penalty_slots(H)
    constexpr uint32_t kNone = 0xFFFFFFFFu;
    const int tid = threadIdx.x;
    const int Smax = penalty_slots(a.H);
    uint32_t* keys = sm;
    uint32_t* cnt = sm + Smax;
    for (int64_t row = blockIdx.x; row < a.B; row += gridDim.x) {
        const float r = a.rep ? a.rep[row] : 1.f;
        const float f = a.freq ? a.freq[row] : 0.f;
        const float rho = a.pres ? a.pres[row] : 0.f;
        const bool ok = isfinite(r) && r > 0.f && isfinite(f) && isfinite(rho);
        if (tid == 0 && a.out_status) a.out_status[row] = ok ? kRowOk : kRowBadParam;
        if (!ok) continue;  // the row is left unchanged
        int64_t n64 = a.hist_len ? (int64_t)a.hist_len[row] : a.H;
        n64 = n64 < 0 ? 0 : (n64 > a.H ? a.H : n64);
        const int n = (int)n64;
        if (n == 0) continue;
        const int S = penalty_slots(n);  // <= Smax
        const int sh = 33 - __ffs(S);    // 32 - log2(S)
        for (int j = tid; j < S; j += kPenaltyThreads) {
            keys[j] = kNone;
            cnt[j] = 0;
        }
        __syncthreads();
        const int32_t* h = a.hist + row * a.ldh;
        const int lane = tid & 31;
        // kBatch history entries per thread are loaded before any is counted, so their latencies
        // overlap; whole warps run each batch together (the match needs every lane).
        for (int base = 0; base < n; base += kBatch * kPenaltyThreads) {
            int32_t v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int j = base + u * kPenaltyThreads + tid;
                v[u] = (j < n) ? h[j] : -1;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (base + u * kPenaltyThreads >= n) break;  // uniform across the CTA
                const bool valid = v[u] >= 0 && (int64_t)v[u] < a.V;
                const uint32_t t = valid ? (uint32_t)v[u] : kNone;
                const uint32_t peers = __match_any_sync(0xFFFFFFFFu, t);
                if (valid && lane == __ffs(peers) - 1) count_id(keys, cnt, t, (uint32_t)__popc(peers), S, sh);
            }
        }
        __syncthreads();
        // Every occupied slot rewrites its token: a thread's slots are read first, then written.
        TIn* zrow = static_cast<TIn*>(a.logits) + row * a.ld;
        for (int base = 0; base < S; base += kBatch * kPenaltyThreads) {
            uint32_t t[kBatch];
            float x[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int j = base + u * kPenaltyThreads + tid;
                t[u] = (j < S) ? keys[j] : kNone;
                x[u] = (t[u] != kNone) ? pen_load(zrow + t[u]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (t[u] == kNone) continue;
                const float c = (float)cnt[base + u * kPenaltyThreads + tid];
                const float y = (x[u] > 0.f) ? __fdiv_rn(x[u], r) : __fmul_rn(x[u], r);
                const float s = __fadd_rn(__fmul_rn(f, c), rho);
                pen_store(zrow + t[u], __fsub_rn(y, s));
            }
        }
        __syncthreads();  // the next row reuses the table
    }
}

// Launch over `sms` SMs (defined with the kernel's instantiations).
cudaError_t launch_penalties(const PenaltyArgs& a, bool bf16, int sms, cudaStream_t stream);

}  // namespace tps
