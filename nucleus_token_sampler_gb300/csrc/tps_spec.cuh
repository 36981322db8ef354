// tps_spec.cuh -- speculative acceptance on truncated distributions, one CTA per row.
//
// "Top-p (Nucleus) Sampling, in depth", 'Logprobs, speculative decoding and reproducibility': a
// draft token x is accepted with probability min(1, P(x)/Q(x)) and a rejection draws from the
// normalised positive part of P - Q, which reproduces P exactly; P must be the target's truncated,
// renormalised distribution and Q the distribution the draft actually sampled from.  Here both are
// the sampler's own kept distributions: each row's target and draft logits go through the same
// chain (temperature -> min-p -> top-k -> top-p) under their own parameters, resolved exactly by the
// general path (a kept set, i.e. a cutoff logit, and its fixed-point mass Z), so that
//   P(i) = round(e^-(zmax - z_i)/T 2^44) / Z   for kept i, else 0     (one-hot for a greedy row),
// the very masses a sampling call renormalises.  Then, per row:
//   accepted  iff  u Q(x) < P(x)  (in double), u the acceptance uniform;
//   otherwise the token is argmax over i with r_i = P(i) - Q(i) > 0 of ln r_i - ln(-ln u_i), an
//   exponential race over the residual (lowest index on equal keys).
// Uniforms: Philox4x32-10 keyed by the row's seed at counter (i / 4, row | 2^31, step), word i mod 4,
// mapped to (2 (w >> 9) + 1) 2^-24; token 2^20 - 1 (above every token index) gives the acceptance
// uniform.  Bit 31 of the row word keeps these counters apart from every other draw's.
#pragma once

#include "tps_common.cuh"

namespace tps {

struct SpecArgs {
    const void* target;  // [B, ld] logits of the target model
    const void* draft;   // [B, ld] logits of the draft model
    int64_t B, V, ld;
    const float* tT;     // the target's temperature, top-k, top-p, min-p per row
    const int32_t* tK;
    const float* tP;
    const float* tM;
    const float* dT;     // the draft's
    const int32_t* dK;
    const float* dP;
    const float* dM;
    const int32_t* draft_token;
    const uint64_t* seed;
    uint64_t step;
    int32_t* out_token;
    int32_t* out_accepted;  // nullable
    int32_t* out_status;    // nullable
};

constexpr uint32_t kSpecAcceptSlot = 0xFFFFFu;  // token index of the acceptance uniform

__device__ __forceinline__ double spec_uniform(uint64_t seed, uint32_t row, uint64_t step, uint32_t token)
{
    const uint4 x = philox_block(make_uint4(token >> 2, row | 0x80000000u, (uint32_t)step, (uint32_t)(step >> 32)),
                                 (uint32_t)seed, (uint32_t)(seed >> 32));
    return (double)uniform_grid(pick_word(x, token & 3u)) * 0x1p-24;
}

// One side (target or draft) of a row, resolved.  Its kept set: every finite logit whose key is at
// least key_cut (a greedy side: the token `arg` alone); its fixed-point mass: zk.
struct Side {
    int32_t status;
    bool greedy;
    int32_t arg;
    RowCtx r;
    uint32_t key_cut;
    uint64_t zk;
    const unsigned char* rowp;
};

// The probability a resolved side gives token i whose logit is z (double; exact ratio of the
// fixed-point masses the kept set sums).
__device__ __forceinline__ double side_prob(const Side& sd, int32_t i, float z)
{
    if (sd.greedy) return i == sd.arg ? 1.0 : 0.0;
    if (!(z > -INFINITY) || fkey(z) < sd.key_cut) return 0.0;
    return (double)qmass_d(dist(sd.r, z)) / (double)sd.zk;
}

// A row of `logits` as the general path's source: the aligned interior through 16-byte loads, the
// ragged head and tail in s.xz / s.xi.  Every thread of the CTA calls it.
template <typename TIn>
__device__ GlobalRow<TIn> spec_source(const void* logits, int64_t row, int64_t V, int64_t ld, Shared& s)
{
    constexpr int ES = Elem<TIn>::kBytes;
    const unsigned char* rowp = static_cast<const unsigned char*>(logits) + row * ld * ES;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(rowp), g1 = g0 + (uintptr_t)V * ES;
    uintptr_t a0 = (g0 + 15) & ~(uintptr_t)15, a1 = g1 & ~(uintptr_t)15;
    int nhead, ntail;
    if (a1 <= a0) {
        a0 = a1 = g1;
        nhead = (int)V;
        ntail = 0;
    } else {
        nhead = (int)((a0 - g0) / ES);
        ntail = (int)((g1 - a1) / ES);
    }
    cta_sync();  // the previous user of s.xz / s.nx is done
    const int nx = nhead + ntail;
    if ((int)threadIdx.x < nx) {
        const int32_t xi = ((int)threadIdx.x < nhead) ? (int32_t)threadIdx.x : (int32_t)(V - ntail + (threadIdx.x - nhead));
        s.xz[threadIdx.x] = Elem<TIn>::load1(rowp, xi);
        s.xi[threadIdx.x] = xi;
    }
    if (threadIdx.x == 0) s.nx = nx;
    cta_sync();
    GlobalRow<TIn> src;
    src.vec = reinterpret_cast<const uint4*>(a0);
    src.nvec = (int)((a1 - a0) / 16);
    src.elem0 = nhead;
    return src;
}

// Resolve one side of a row: its maximum and status, and for a sampling side the exact kept set
// and mass through the general path (whose own race is not used).  Every thread calls it.
template <typename TIn>
__device__ Side resolve_side(const void* logits, int64_t row, const SpecArgs& a, float T, int32_t K, float P, float MP,
                             Shared& s)
{
    Side sd;
    const GlobalRow<TIn> src = spec_source<TIn>(logits, row, a.V, a.ld, s);
    sd.rowp = static_cast<const unsigned char*>(logits) + row * a.ld * Elem<TIn>::kBytes;
    float m = -INFINITY;
    src.for_each(s, [&](float z, int32_t) { m = fmax_nan(m, z); });
    m = warp_max_nan(m);
    cta_sync();
    if ((threadIdx.x & 31) == 0) s.rf[threadIdx.x >> 5] = m;
    cta_sync();
    float zmax = s.rf[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) zmax = fmax_nan(zmax, s.rf[w]);
    sd.greedy = false;
    sd.arg = -1;
    sd.key_cut = 0;
    sd.zk = 0;
    sd.status = kRowOk;
    if (isnan(zmax) || zmax == INFINITY) sd.status = kRowNan;
    else if (!(isfinite(T) && isfinite(P) && isfinite(MP))) sd.status = kRowBadParam;
    else if (zmax == -INFINITY) sd.status = kRowAllMasked;
    const float minp = (MP > 0.f) ? fminf(MP, 1.f) : 0.f;
    sd.r = make_ctx(zmax, T > 0.f ? T : 1.f, minp);
    if (sd.status != kRowOk) return sd;
    if (T <= 0.f) {  // greedy: the lowest index of the maximum, probability 1
        uint32_t mi = 0xFFFFFFFFu;
        src.for_each(s, [&](float z, int32_t i) {
            if (z == zmax) mi = min(mi, (uint32_t)i);
        });
        sd.greedy = true;
        sd.arg = (int32_t)block_min_u32(mi, s);
        return sd;
    }
    const float zc = minp_threshold(sd.r);
    RaceCtx rc;
    rc.k0 = (uint32_t)a.seed[row];
    rc.k1 = (uint32_t)(a.seed[row] >> 32);
    rc.row = (uint32_t)row;
    rc.s_lo = (uint32_t)a.step;
    rc.s_hi = (uint32_t)(a.step >> 32);
    SoloTopo topo;
    const RowResult res = general_path(topo, s, src, sd.r, zc, (K > 0) && ((int64_t)K < a.V), K, P, rc, nullptr, true);
    sd.key_cut = res.key_cut;
    sd.zk = res.zk;
    return sd;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads) spec_rows_kernel(const SpecArgs a)
{
    extern __shared__ __align__(128) unsigned char dsmem[];
    Shared& s = *reinterpret_cast<Shared*>(dsmem);
    const int tid = threadIdx.x;
    for (int64_t row = blockIdx.x; row < a.B; row += gridDim.x) {
        const Side st = resolve_side<TIn>(a.target, row, a, a.tT[row], a.tK[row], a.tP[row], a.tM[row], s);
        const Side sq = resolve_side<TIn>(a.draft, row, a, a.dT[row], a.dK[row], a.dP[row], a.dM[row], s);
        const int32_t x = a.draft_token[row];
        const uint64_t seed = a.seed[row];
        int32_t status = st.status != kRowOk ? st.status : sq.status;
        double px = 0.0, qx = 0.0;
        if (status == kRowOk) {
            if (x < 0 || (int64_t)x >= a.V) {
                status = kRowBadParam;
            } else {
                px = side_prob(st, x, Elem<TIn>::load1(st.rowp, x));
                qx = side_prob(sq, x, Elem<TIn>::load1(sq.rowp, x));
                if (!(qx > 0.0)) status = kRowBadParam;  // the draft cannot have drawn x
            }
        }
        int32_t token = -1, accepted = 0;
        if (status == kRowOk) {
            const double u = spec_uniform(seed, (uint32_t)row, a.step, kSpecAcceptSlot);
            if (u * qx < px) {
                accepted = 1;
                token = x;
            } else {
                // the residual race over the target's kept tokens with P(i) > Q(i); a token is
                // skipped before its uniform is drawn when even the largest -ln(-ln u) of the
                // uniform grid (16.6355...) cannot lift ln P(i) to this thread's best key
                const GlobalRow<TIn> src = spec_source<TIn>(a.target, row, a.V, a.ld, s);
                ArgBest best;
                best.key = -INFINITY;
                best.idx = 0x7FFFFFFF;
                src.for_each(s, [&](float z, int32_t i) {
                    const double pi = side_prob(st, i, z);
                    if (!(pi > 0.0)) return;
                    if ((double)logf((float)pi) + 16.64 < best.key - 1e-3) return;
                    const double qi = side_prob(sq, i, Elem<TIn>::load1(sq.rowp, i));
                    const double r = pi - qi;
                    if (!(r > 0.0)) return;
                    const double key = log(r) - log(-log(spec_uniform(seed, (uint32_t)row, a.step, (uint32_t)i)));
                    if (better(key, i, best.key, best.idx)) {
                        best.key = key;
                        best.idx = i;
                    }
                });
                token = block_argbest(best, s).idx;
                if (token == 0x7FFFFFFF) {  // no residual above rounding: P and Q agree, x stands
                    token = x;
                    accepted = 1;
                }
            }
        }
        if (tid == 0) {
            a.out_token[row] = token;
            if (a.out_accepted) a.out_accepted[row] = accepted;
            if (a.out_status) a.out_status[row] = status;
        }
        cta_sync();
    }
}

cudaError_t launch_spec(const SpecArgs& a, bool bf16, int sms, cudaStream_t stream);

}  // namespace tps
