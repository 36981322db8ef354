// tps_device.cuh -- small device helpers for the sampler kernels (sm_103a).
//
// Philox4x32-10, order-preserving float keys, the fixed-point mass of a token, bulk-copy and
// mbarrier wrappers (inline PTX), and warp/block reductions.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace tps {

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).  Ten rounds; each round multiplies the
// even counter words by two fixed 32-bit constants, mixes the high halves with the odd words and
// the key, and the key advances by the two Weyl increments between rounds.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_hi = __umulhi(kMulA, c.x), a_lo = kMulA * c.x;
        const uint32_t b_hi = __umulhi(kMulB, c.z), b_lo = kMulB * c.z;
        c = make_uint4(b_hi ^ c.y ^ k0, b_lo, a_hi ^ c.w ^ k1, a_lo);
        k0 += kWeylA;
        k1 += kWeylB;
    }
    return c;
}

// Two blocks at once, their rounds interleaved: each block's ten rounds are a chain of dependent
// multiplies, so two independent chains keep the multiplier busy for twice the work in about the
// same latency.  Bit for bit the same function as philox4x32_10 on each counter.
__device__ __forceinline__ void philox4x32_10_x2(uint4& c, uint4& d, uint32_t k0, uint32_t k1)
{
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_hi = __umulhi(kMulA, c.x), a_lo = kMulA * c.x;
        const uint32_t b_hi = __umulhi(kMulB, c.z), b_lo = kMulB * c.z;
        const uint32_t e_hi = __umulhi(kMulA, d.x), e_lo = kMulA * d.x;
        const uint32_t f_hi = __umulhi(kMulB, d.z), f_lo = kMulB * d.z;
        c = make_uint4(b_hi ^ c.y ^ k0, b_lo, a_hi ^ c.w ^ k1, a_lo);
        d = make_uint4(f_hi ^ d.y ^ k0, f_lo, e_hi ^ d.w ^ k1, e_lo);
        k0 += kWeylA;
        k1 += kWeylB;
    }
}

// One block out of line: the race code that draws it stays small inside unrolled loops.
static __device__ __noinline__ uint4 philox_block(uint4 c, uint32_t k0, uint32_t k1) { return philox4x32_10(c, k0, k1); }

// Uniform in (0, 1): an odd multiple of 2^-24, exact in float and double.
__device__ __forceinline__ uint32_t uniform_grid(uint32_t x) { return 2u * (x >> 9) + 1u; }

__device__ __forceinline__ uint32_t pick_word(uint4 v, uint32_t w)
{
    return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------------------------
// Order-preserving 32-bit key of a float (larger float -> larger key).  -0.0 is folded onto
// +0.0 first so equal logits always share a key.  -inf maps below every finite value.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t fkey(float z)
{
    uint32_t b = __float_as_uint(z);
    b = (b == 0x80000000u) ? 0u : b;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k)
{
    const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

// ---------------------------------------------------------------------------------------------
// Row constants shared by every pass.
// ---------------------------------------------------------------------------------------------
struct RowCtx {
    float zmax;     // largest finite logit
    float invT;     // 1 / T, clamped to FLT_MAX
    float T;        // temperature (> 0 on the sampling path)
    float minp;     // min_p clamped to [0, 1]; 0 = off
    float L_lo;     // -ln(minp) minus a safety margin: d below this always survives min-p
    float L_hi;     // -ln(minp) plus the margin: d above this never survives
};

// Scaled distance from the maximum, d = (zmax - z) / T >= 0, monotone non-increasing in z.
__device__ __forceinline__ float dist(const RowCtx& r, float z) { return (r.zmax - z) * r.invT; }

// round(e * 2^44) to the nearest integer, ties to even, for 0 <= e <= 1, as hi * 2^22 + lo -- with
// float adds and one fused multiply-add instead of a float-to-64-bit conversion (a slow pipe):
//   t  = e 2^22 + 2^23 rounded down = 2^23 + floor(e 2^22) exactly (results are integers there);
//   lo = e 2^44 - floor(e 2^22) 2^22 is exact in one fma and lies in [0, 2^22); adding 2^23 rounds
//        it to the nearest integer, ties to even.
// hi 2^22 is an even integer, so adding it back cannot change the direction of a tie.
struct Fixed44 {
    uint32_t hi, lo;
};
__device__ __forceinline__ Fixed44 fixed44_parts(float e)
{
    const float t = __fadd_rd(e * 0x1p22f, 0x1p23f);
    const float rem = __fmaf_rn(-__fsub_rn(t, 0x1p23f), 0x1p22f, e * 0x1p44f);
    Fixed44 f;
    f.hi = __float_as_uint(t) - 0x4B000000u;
    f.lo = __float_as_uint(__fadd_rn(rem, 0x1p23f)) - 0x4B000000u;
    return f;
}
__device__ __forceinline__ uint64_t fixed44(float e)
{
    const Fixed44 f = fixed44_parts(e);
    return ((uint64_t)f.hi << 22) + f.lo;
}

// Fixed-point mass of a token: round(exp(-d) * 2^44) as an integer.  Sums of these are exact,
// order-independent and deterministic; a row of up to 2^20 tokens cannot overflow 64 bits.
__device__ __forceinline__ uint64_t qmass_d(float d) { return fixed44(expf(-d)); }

// The double-precision min-p decision (the same operations as the float64 definition), out of
// line: it runs only for tokens within a narrow margin of the cut, and inlining it into every
// element of an unrolled loop would crowd the instruction cache.
static __device__ __noinline__ bool minp_ok_double(float zmax, float T, float minp, float z)
{
    const double dd = __ddiv_rn(__dsub_rn((double)zmax, (double)z), (double)T);
    return exp(-dd) >= (double)minp;
}

// min-p survival, p_i >= min_p * p_max, i.e. exp(-(zmax - z) / T) >= min_p.  Decided in float
// away from the cut, and in double within a margin of it, so the decision matches an exact double
// evaluation.
__device__ __forceinline__ bool minp_ok(const RowCtx& r, float z, float d)
{
    if (!(r.minp > 0.f)) return true;
    if (d < r.L_lo) return true;
    if (d > r.L_hi) return false;
    return minp_ok_double(r.zmax, r.T, r.minp, z);
}

// ---------------------------------------------------------------------------------------------
// Element loads.
// ---------------------------------------------------------------------------------------------
template <typename TIn> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    static constexpr int kBytes = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&z)[kPerVec])
    {
        z[0] = __uint_as_float(v.x);
        z[1] = __uint_as_float(v.y);
        z[2] = __uint_as_float(v.z);
        z[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static float load1(const void* p, int64_t i)
    {
        return __ldg(reinterpret_cast<const float*>(p) + i);
    }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    static constexpr int kBytes = 2;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&z)[kPerVec])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            z[2 * j] = __uint_as_float(w[j] << 16);
            z[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static float load1(const void* p, int64_t i)
    {
        const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p) + i);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};

// ---------------------------------------------------------------------------------------------
// Bulk copy global -> own shared memory, completed on an mbarrier (no multicast).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Order this thread's earlier generic-proxy accesses of shared memory before later async-proxy
// (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One bounded probe of phase `parity`: the thread is suspended (not spinning) until the phase
// completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 0)
{
    uint32_t ok;
    if (hint_ns) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
    }
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` for at most `limit_ns` nanoseconds.  Returns false on timeout.
// Each probe suspends the thread for up to 20 us, so a waiting warp does not take issue slots from
// the warps that are computing.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Split cluster barrier: arrive (release this CTA's prior shared-memory writes and reads), wait
// (acquire).  Every thread of every CTA of the cluster executes both, in order.
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// max with NaN propagation (a NaN anywhere in the row survives the reduction).
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Three-input float maximum with NaN propagation (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3_nan(float a, float b, float c)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Lane-wise maximum of two packed bfloat16 pairs with NaN propagation.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// ---------------------------------------------------------------------------------------------
// Warp reductions.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max_nan(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v)
{
    return __reduce_min_sync(0xFFFFFFFFu, v);
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v)
{
    return __reduce_max_sync(0xFFFFFFFFu, v);
}
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v)
{
    return __reduce_add_sync(0xFFFFFFFFu, v);
}
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// (key, index) argmax with the lowest index winning equal keys.
struct ArgBest {
    double key;
    int32_t idx;
};
__device__ __forceinline__ bool better(double ka, int32_t ia, double kb, int32_t ib)
{
    return ka > kb || (ka == kb && (uint32_t)ia < (uint32_t)ib);
}
__device__ __forceinline__ ArgBest warp_argbest(ArgBest a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double k = __shfl_xor_sync(0xFFFFFFFFu, a.key, o);
        const int32_t i = __shfl_xor_sync(0xFFFFFFFFu, a.idx, o);
        if (better(k, i, a.key, a.idx)) {
            a.key = k;
            a.idx = i;
        }
    }
    return a;
}

}  // namespace tps
