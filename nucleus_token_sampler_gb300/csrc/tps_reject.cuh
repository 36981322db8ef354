// tps_reject.cuh -- the sort-free rejection draw, one CTA per row.
//
// "Top-p (Nucleus) Sampling, in depth", 'Sort-free top-p by rejection sampling': a token belongs to
// the nucleus exactly when the mass of strictly more probable tokens is below p, so a draw can be
// tested with one reduction over the vocabulary instead of a sort; a rejected draw raises the pivot
// and discards the rejected token with everything less probable, and because the nucleus always lies
// above the pivot, accepted tokens follow the renormalised nucleus distribution.  Here, per row:
//   S    = the survivors of min-p and top-k (an upper set in z), Z_S their fixed-point mass;
//   round r (r = 0, 1, ...): race among the survivors above the pivot (all of S in round 0) in
//        proportion to e^-(zmax - z)/T -- argmax of -(zmax - z_i)/T - ln(-ln u_i) with round r's
//        uniforms, lowest index on equal keys -- and accept the winner t when it is in the class of
//        the maximum, when p >= 1, or when the fixed-point mass of the survivors with a larger logit
//        is below p Z_S (the test that defines the nucleus); otherwise t's logit becomes the pivot.
// Round r's uniforms are the race's generator and mapping with r + 1 in bits 18..31 of the counter's
// first word: Philox4x32-10 keyed by the row's seed at counter ((i / 4) | (r + 1) << 18, row, step),
// word i mod 4.  Since i / 4 < 2^18 for V <= 2^20, no round reuses the select path's uniforms.  The
// kept set reported (cutoff, count) is the select path's; only the draw differs.
#pragma once

#include "tps_common.cuh"

namespace tps {

constexpr uint32_t kMaxRounds = 4096;  // a bound on the rounds (each rejection drops a whole class)

struct RejectArgs {
    Args a;              // the sampling call's arguments (out_probs, logprobs and top tokens unused)
    int32_t* out_rounds;  // [B] or null: rounds the row took (0 for greedy and failed rows)
};

__device__ __forceinline__ float round_u(const RaceCtx& rc, uint32_t round, int32_t i)
{
    const uint4 x = philox_block(make_uint4(((uint32_t)i >> 2) | ((round + 1u) << 18), rc.row, rc.s_lo, rc.s_hi),
                                 rc.k0, rc.k1);
    return (float)uniform_grid(pick_word(x, (uint32_t)i & 3u)) * 0x1p-24f;
}

// The race of one round over the survivors with a logit above zpiv (every thread of the CTA calls it).
// Float keys rank the tokens; when the best leads the second by less than the float/double margin,
// every token within the margin is re-evaluated in double precision exactly as the definition does.
template <typename Src, typename InS>
__device__ int32_t round_race(Shared& s, const Src& src, const RowCtx& r, const RaceCtx& rc, uint32_t round, float zpiv,
                              float dlow, InS&& in_s)
{
    Top2 t2;
    t2.init();
    src.for_each(s, [&](float z, int32_t i) {
        if (!(z > zpiv) || !in_s(z)) return;
        const float d = dist(r, z);
        if (16.64f - d < t2.k2) return;  // cannot be among this thread's two best
        t2.add(race_key32(d, round_u(rc, round, i)), i);
    });
    t2 = warp_top2(t2);
    cta_sync();
    if ((threadIdx.x & 31) == 0) {
        s.rab[threadIdx.x >> 5].key = (double)t2.k1;
        s.rab[threadIdx.x >> 5].idx = t2.i1;
        s.rf[threadIdx.x >> 5] = t2.k2;
    }
    cta_sync();
    Top2 b;
    b.init();
    for (int w = 0; w < kWarps; ++w) {
        Top2 x;
        x.k1 = (float)s.rab[w].key;
        x.i1 = s.rab[w].idx;
        x.k2 = s.rf[w];
        b.merge(x);
    }
    const float tol = race_tol(dlow);
    if (b.k1 - b.k2 > tol) return b.i1;
    ArgBest mine;
    mine.key = -INFINITY;
    mine.idx = 0x7FFFFFFF;
    src.for_each(s, [&](float z, int32_t i) {
        if (!(z > zpiv) || !in_s(z)) return;
        const float u = round_u(rc, round, i);
        if (race_key32(dist(r, z), u) >= b.k1 - tol) {
            const double k64 = race_key64(r, z, u);
            if (better(k64, i, mine.key, mine.idx)) {
                mine.key = k64;
                mine.idx = i;
            }
        }
    });
    return block_argbest(mine, s).idx;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads) reject_rows_kernel(const RejectArgs ra)
{
    extern __shared__ __align__(128) unsigned char dsmem[];
    Shared& s = *reinterpret_cast<Shared*>(dsmem);
    const Args& a = ra.a;
    const int tid = threadIdx.x;
    constexpr int ES = Elem<TIn>::kBytes;
    for (int64_t row = blockIdx.x; row < a.B; row += gridDim.x) {
        // the row as a source: aligned interior through 16-byte loads, ragged head and tail in s.xz
        const unsigned char* rowp = static_cast<const unsigned char*>(a.logits) + row * a.ld * ES;
        const uintptr_t g0 = reinterpret_cast<uintptr_t>(rowp), g1 = g0 + (uintptr_t)a.V * ES;
        uintptr_t a0 = (g0 + 15) & ~(uintptr_t)15, a1 = g1 & ~(uintptr_t)15;
        int nhead, ntail;
        if (a1 <= a0) {
            a0 = a1 = g1;
            nhead = (int)a.V;
            ntail = 0;
        } else {
            nhead = (int)((a0 - g0) / ES);
            ntail = (int)((g1 - a1) / ES);
        }
        cta_sync();
        if (tid < nhead + ntail) {
            const int32_t xi = (tid < nhead) ? tid : (int32_t)(a.V - ntail + (tid - nhead));
            s.xz[tid] = Elem<TIn>::load1(rowp, xi);
            s.xi[tid] = xi;
        }
        if (tid == 0) s.nx = nhead + ntail;
        cta_sync();
        GlobalRow<TIn> src;
        src.vec = reinterpret_cast<const uint4*>(a0);
        src.nvec = (int)((a1 - a0) / 16);
        src.elem0 = nhead;

        const float T = a.temperature[row], P = a.top_p[row], MP = a.min_p[row];
        const int32_t K = a.top_k[row];
        const uint64_t seed = a.seed[row];
        float m = -INFINITY;
        src.for_each(s, [&](float z, int32_t) { m = fmax_nan(m, z); });
        m = warp_max_nan(m);
        cta_sync();
        if ((tid & 31) == 0) s.rf[tid >> 5] = m;
        cta_sync();
        float zmax = s.rf[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) zmax = fmax_nan(zmax, s.rf[w]);
        int32_t status = kRowOk;
        if (isnan(zmax) || zmax == INFINITY) status = kRowNan;
        else if (!(isfinite(T) && isfinite(P) && isfinite(MP))) status = kRowBadParam;
        else if (zmax == -INFINITY) status = kRowAllMasked;
        const float qnan = __uint_as_float(0x7FC00000u);
        if (status != kRowOk) {
            if (tid == 0) {
                write_row(a, row, -1, status, qnan, 0);
                if (ra.out_rounds) ra.out_rounds[row] = 0;
            }
            continue;
        }
        if (T <= 0.f) {  // greedy: the lowest index of the maximum; no draw
            uint32_t mi = 0xFFFFFFFFu;
            src.for_each(s, [&](float z, int32_t i) {
                if (z == zmax) mi = min(mi, (uint32_t)i);
            });
            mi = block_min_u32(mi, s);
            if (tid == 0) {
                write_row(a, row, (int32_t)mi, kRowOk, zmax, 1);
                if (ra.out_rounds) ra.out_rounds[row] = 0;
            }
            continue;
        }
        const float minp = (MP > 0.f) ? fminf(MP, 1.f) : 0.f;
        const RowCtx r = make_ctx(zmax, T, minp);
        const float zc = minp_threshold(r);
        const bool topk_on = (K > 0) && ((int64_t)K < a.V);
        RaceCtx rc;
        rc.k0 = (uint32_t)seed;
        rc.k1 = (uint32_t)(seed >> 32);
        rc.row = (uint32_t)row;
        rc.s_lo = (uint32_t)a.step;
        rc.s_hi = (uint32_t)(a.step >> 32);
        SoloTopo topo;
        // S and its mass (top-p off), then the nucleus the select path reports (its own race unused)
        const RowResult rs = general_path(topo, s, src, r, zc, topk_on, K, 1.f, rc, nullptr, true);
        const RowResult rk = (P < 1.f) ? general_path(topo, s, src, r, zc, topk_on, K, P, rc, nullptr, false) : rs;
        const uint32_t key_s = rs.key_cut;
        auto in_s = [&](float z) { return z > -INFINITY && fkey(z) >= key_s; };
        const double tmass = (double)P * (double)rs.zk;
        const float dlow = dist(r, key_to_float(key_s));
        float zpiv = -INFINITY;
        int32_t token = -1;
        uint32_t round = 0;
        for (; round < kMaxRounds; ++round) {
            const int32_t t = round_race(s, src, r, rc, round, zpiv, dlow, in_s);
            const float zt = Elem<TIn>::load1(rowp, t);
            if (zt == zmax || !(P < 1.f)) {
                token = t;
                break;
            }
            // the fixed-point mass of the survivors with a larger logit than t's
            uint64_t hi = 0, lo = 0;
            src.for_each(s, [&](float z, int32_t) {
                if (z > zt && in_s(z)) {
                    const Fixed44 f = fixed44_parts(expf(-dist(r, z)));
                    hi += f.hi;
                    lo += f.lo;
                }
            });
            const uint64_t above = block_sum_u64((hi << 22) + lo, s);
            if ((double)above < tmass) {
                token = t;
                break;
            }
            zpiv = zt;
        }
        if (tid == 0) {
            write_row(a, row, token, token >= 0 ? kRowOk : kRowTimeout, key_to_float(rk.key_cut), (int32_t)rk.nk);
            if (ra.out_rounds) ra.out_rounds[row] = (int32_t)min(round + 1u, kMaxRounds);
        }
    }
}

cudaError_t launch_reject(const RejectArgs& ra, bool bf16, int sms, cudaStream_t stream);

}  // namespace tps
