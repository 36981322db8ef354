/*
 * tps.h -- C ABI of the GB300 batched token sampler.
 *
 * For each row b of a [B, V] logits matrix the library applies, in this fixed order,
 *   temperature -> min-p -> top-k -> top-p (nucleus) -> renormalise -> sample one token,
 * as described on the pages "What do temperature, top-k and top-p each do to the next-token
 * distribution, and in what order does a serving engine apply them?" ('A strong answer': the
 * p_i(T) equation, the engine order and the exponential-race draw) and "Implement batched top-p
 * sampling with temperature" ('How to approach it': keep token i iff the mass of strictly more
 * probable tokens is below p; 'A strong answer': the greedy branch and per-request p).
 * An optional stage ahead of that chain, tps_apply_penalties, applies repetition, frequency and
 * presence penalties to the raw logits in place.
 *
 * Rules, per row (T = temperature[b], k = top_k[b], p = top_p[b], m = min_p[b]):
 *   - T <= 0: greedy; the token is the lowest index holding the largest logit.
 *   - min-p keeps tokens with p_i >= m * p_max (m <= 0: off; m > 1 acts as 1).
 *   - top-k keeps tokens with fewer than k strictly larger logits, so ties at the k-th value all
 *     survive (k <= 0 or k >= V: off).
 *   - top-p keeps token i of the survivors S iff the mass of the survivors with a strictly larger
 *     logit, renormalised over S, is below p.  The class of the largest logit is always kept;
 *     p >= 1 keeps S; p <= 0 keeps only that class.
 *   - -inf logits get probability 0 and are never kept.
 *   - the token is argmax over the kept set of  -(zmax - z_i)/T - ln(-ln u_i)  (an exponential race,
 *     argmax P_i / E_i), lowest index on equal keys, with
 *     u_i = (2 * (x >> 9) + 1) * 2^-24 and x = word (i mod 4) of Philox4x32-10 with key = seed[b]
 *     (low word first) and counter = (i / 4, b, step low word, step high word).
 *
 * Calling convention (all entry points):
 *   - every pointer argument is a DEVICE pointer owned by the caller, except where marked;
 *   - a sampling call that runs the streaming kernel (tps_sample, tps_sample_ex, tps_sample_kernel
 *     and tps_sample_full, see tps_kernel) draws a small scratch buffer (claim counters, a row
 *     list and, for a batch of fewer than four rows per SM, the partial results of its split rows:
 *     a few KB for 1,024 rows of 128,256 logits, at most about 2.5 MB for a split batch) from a
 *     stream-ordered memory pool the library creates once per device, and returns it on the call's
 *     stream; the pool keeps up to 64 MiB reserved between calls.  tps_sample_noalloc uses a fixed
 *     array instead; no other call allocates device memory;
 *   - the library never synchronises the host, keeps no state between calls beyond that pool and
 *     a per-device cache of queried limits, and may be called from several host threads at once;
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); all work is enqueued on it;
 *   - the return value is a tps_status; errors in the arguments are reported before anything is
 *     enqueued; problems in a row's data are reported per row in out_status and never abort the
 *     batch (a failed row gets token -1, cutoff NaN, kept 0 and an all-zero probability row).
 */
#ifndef TPS_H_
#define TPS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the logits matrix. */
typedef enum { TPS_F32 = 0, TPS_BF16 = 1 } tps_dtype;

/* Synchronous return codes. */
typedef enum {
    TPS_OK = 0,
    TPS_ERR_ARG = 1,           /* a required pointer is NULL, B < 0, V < 1 or ld < V            */
    TPS_ERR_DTYPE = 2,         /* dtype is not a tps_dtype                                      */
    TPS_ERR_UNSUPPORTED_V = 3, /* V is above tps_max_vocab(dtype)                               */
    TPS_ERR_ALIGN = 4,         /* logits, out_probs or a parameter array is not element-aligned */
    TPS_ERR_CUDA = 5,          /* the CUDA runtime refused the launch (see tps_last_cuda_error) */
    TPS_ERR_SCRATCH = 6        /* tps_sample_noalloc: the call needs more than its fixed scratch   */
} tps_status;

/* Per-row outcome written to out_status. */
typedef enum {
    TPS_ROW_OK = 0,
    TPS_ROW_NAN = 1,        /* the row holds a NaN or +inf logit ("Top-p (Nucleus) Sampling, in
                               depth", 'Failure modes': fail the request rather than sample)    */
    TPS_ROW_ALL_MASKED = 2, /* every logit is -inf                                              */
    TPS_ROW_BAD_PARAM = 3,  /* temperature, top_p or min_p is NaN or infinite                    */
    TPS_ROW_TIMEOUT = 4     /* a bounded wait inside the kernel gave up; the row was not sampled */
} tps_row_status;

/*
 * tps_sample -- sample one token per row of a dense [B, V] logits matrix.
 *
 *   logits       [B, V] row-major, TPS_F32 (float) or TPS_BF16 (bfloat16); element-aligned.
 *   dtype        a tps_dtype.
 *   B, V         rows and vocabulary size; B = 0 returns TPS_OK and enqueues nothing.
 *   temperature  [B] float.     top_k [B] int32.     top_p [B] float.     min_p [B] float.
 *   seed         [B] uint64 Philox key per row.
 *   step         64-bit counter word shared by the batch (advance it every decode step).
 *   out_token    [B] int32: the sampled token id, or -1 for a failed row.
 *   out_probs    [B, V] float, or NULL: the renormalised distribution the token was drawn from
 *                (0 outside the kept set; one-hot for greedy rows).
 *   stream       cudaStream_t.
 */
int tps_sample(const void* logits, int dtype, int64_t B, int64_t V, const float* temperature,
               const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
               uint64_t step, int32_t* out_token, float* out_probs, void* stream);

/*
 * tps_sample_ex -- tps_sample with a row stride and optional diagnostics.
 *
 *   ld           row stride of `logits` in elements (ld >= V); out_probs stays dense [B, V].
 *   out_status   [B] int32 tps_row_status, or NULL.
 *   out_cutoff   [B] float, or NULL: v*, the smallest kept logit.  Token i is kept iff its logit is
 *                finite and >= v* (greedy rows: v* = the largest logit and only the returned token
 *                counts as kept).
 *   out_kept     [B] int32, or NULL: the number of kept tokens (1 for greedy rows).
 */
int tps_sample_ex(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                  const float* temperature, const int32_t* top_k, const float* top_p,
                  const float* min_p, const uint64_t* seed, uint64_t step, int32_t* out_token,
                  float* out_probs, int32_t* out_status, float* out_cutoff, int32_t* out_kept,
                  void* stream);

/*
 * Which kernel samples the rows (tps_sample_kernel).
 *   AUTO    the library's choice (what tps_sample uses): below 32 rows the cluster kernel; from 32
 *           rows the batch is split -- the streaming kernel samples the rows with min-p (and greedy
 *           and failed rows) and lists the others in its scratch, and the cluster kernel, launched
 *           right behind it, samples the listed rows (rows without min-p take the general path,
 *           which makes several passes over the row, and the cluster kernel makes them on-chip).
 *           When no row is listed the cluster kernel finds an empty list and exits.
 *   CLUSTER every row by the cluster kernel (one cluster of up to 16 CTAs per row).
 *   STREAM  every row by the streaming kernel (one CTA per SM, rows streamed through a ring); the
 *           fastest choice for a batch whose rows all use min-p or are greedy, e.g. decode batches
 *           with min-p set, and much slower for rows without min-p.
 */
typedef enum {
    TPS_KERNEL_AUTO = 0,
    TPS_KERNEL_CLUSTER = 1,
    TPS_KERNEL_STREAM = 2
} tps_kernel;

/*
 * tps_sample_kernel -- tps_sample_ex with an explicit kernel choice (same results for every
 * choice; the choice only changes speed).  `kernel` is a tps_kernel; any other value is
 * TPS_ERR_ARG.  TPS_KERNEL_CLUSTER returns TPS_ERR_UNSUPPORTED_V when 16 CTAs cannot hold a row.
 */
int tps_sample_kernel(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                      const float* temperature, const int32_t* top_k, const float* top_p,
                      const float* min_p, const uint64_t* seed, uint64_t step, int32_t* out_token,
                      float* out_probs, int32_t* out_status, float* out_cutoff, int32_t* out_kept,
                      int kernel, void* stream);

/* Most top tokens tps_sample_full reports per row. */
#define TPS_MAX_TOP 32

/*
 * tps_sample_full -- tps_sample_kernel plus processed log-probabilities: those of the sampled
 * token and of the row's most probable kept tokens ("processed": under the renormalised kept
 * distribution that out_probs holds, not the raw softmax; "Top-p (Nucleus) Sampling, in depth",
 * 'Logprobs, speculative decoding and reproducibility': under the processed distribution every
 * token outside the nucleus has probability zero, and callers must know which of the two they get).
 *
 *   out_logprob      [B] float, or NULL: ln P(token) = -(zmax - z_token)/T - ln(sum over kept i of
 *                    e^{-(zmax - z_i)/T}); 0 for greedy rows, NaN for failed rows.
 *   n_top            0 .. TPS_MAX_TOP top tokens per row (0: none, and the two pointers below are
 *                    ignored); any other value is TPS_ERR_ARG.
 *   out_top_idx      [B, n_top] int32 (row-major, caller-owned device memory): the n_top most
 *                    probable kept tokens of each row, by probability descending and then index
 *                    ascending; slots past the row's kept count hold -1.  A greedy row holds its
 *                    token then -1s; a failed row holds -1s.  NULL with n_top > 0 is TPS_ERR_ARG.
 *   out_top_logprob  [B, n_top] float: ln P of those tokens (0 for a greedy row's token, -inf for
 *                    empty slots, NaN for every slot of a failed row).
 * Every other argument is as in tps_sample_kernel.  Asking for top tokens on rows that take the
 * general path (more than 256 survivors) costs one or more extra passes over those rows.
 */
int tps_sample_full(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                    const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                    uint64_t step, int32_t* out_token, float* out_probs, int32_t* out_status, float* out_cutoff,
                    int32_t* out_kept, float* out_logprob, int32_t n_top, int32_t* out_top_idx,
                    float* out_top_logprob, int kernel, void* stream);

/* Longest per-row history tps_apply_penalties takes. */
#define TPS_MAX_HISTORY 8192

/*
 * tps_apply_penalties -- repetition, frequency and presence penalties on raw logits, IN PLACE, the
 * stage that runs ahead of the sampler ("Top-p (Nucleus) Sampling, in depth", "Where top-p sits in
 * the sampler chain"; "What do temperature, top-k and top-p each do ...", "What interviewers probe
 * next": on raw logits, before temperature).  For every token t occurring c_t > 0 times in the row's
 * history:
 *     y = z_t / r  if z_t > 0,  z_t * r  otherwise;      z_t <- y - (f * c_t + rho)
 * computed in float32, one correctly rounded operation at a time in that order, and rounded to
 * nearest-even bfloat16 for bfloat16 logits.  Logits of tokens not in the history are not touched.
 *
 *   logits      [B, ld] float32 or bfloat16 (dtype as in tps_sample), modified in place.
 *   history     [B, ldh] int32 token ids, ldh >= H; ids outside [0, V) are ignored (use -1 to pad).
 *               May be NULL when H == 0.
 *   H           0 .. TPS_MAX_HISTORY entries per row; larger is TPS_ERR_ARG.
 *   hist_len    [B] int32 or NULL: row b uses history entries [0, hist_len[b]) (clamped to [0, H]);
 *               NULL means H for every row.
 *   repetition  [B] float or NULL (1: off); must be finite and > 0.
 *   frequency   [B] float or NULL (0: off); must be finite.
 *   presence    [B] float or NULL (0: off); must be finite.
 *   out_status  [B] int32 or NULL: TPS_ROW_OK, or TPS_ROW_BAD_PARAM for a row whose penalty values
 *               are invalid (that row is left unchanged).
 * All pointers are caller-owned device memory; the call allocates nothing and is stream-ordered on
 * `stream`.  With no penalty array and no out_status it returns TPS_OK and enqueues nothing.
 * Returns TPS_ERR_ARG / _DTYPE / _ALIGN / _UNSUPPORTED_V (V > INT32_MAX) / _CUDA as tps_sample does.
 */
int tps_apply_penalties(void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const int32_t* history,
                        int64_t H, int64_t ldh, const int32_t* hist_len, const float* repetition,
                        const float* frequency, const float* presence, int32_t* out_status, void* stream);

/*
 * tps_sample_rejection -- the same kept set and distribution as tps_sample, drawn by sort-free
 * rejection rounds instead of one race over the kept set ("Top-p (Nucleus) Sampling, in depth",
 * 'Sort-free top-p by rejection sampling': a token is in the nucleus exactly when the mass of
 * strictly more probable tokens is below p, so a draw is tested with one reduction instead of a
 * sort; a rejected draw raises the pivot and drops the rejected token and everything less probable).
 *   S = the survivors of min-p and top-k, Z_S their mass.  Round r races among the survivors above
 *   the pivot (all of S in round 0): argmax of -(zmax - z_i)/T - ln(-ln u_i), lowest index on equal
 *   keys.  The winner t is accepted when it holds the largest logit, when p >= 1, or when the mass of
 *   the survivors with a larger logit is below p Z_S; otherwise its logit becomes the pivot.
 *   Round r's uniforms: as tps_sample's, with r + 1 in bits 18..31 of the counter's first word
 *   (counter ((i / 4) | (r + 1) << 18, b, step low, step high)), so they never coincide with them.
 *   The draw follows the renormalised kept distribution but differs from tps_sample's token.
 *
 *   Arguments as tps_sample_ex (out_status, out_cutoff, out_kept: NULL or [B]; cutoff and kept are
 *   tps_sample's, the nucleus itself), plus out_rounds: NULL or [B] int32, the rounds the row took
 *   (0 for greedy and failed rows).  All pointers are caller-owned device memory; the call allocates
 *   nothing and is stream-ordered on `stream`.
 */
int tps_sample_rejection(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                         const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                         uint64_t step, int32_t* out_token, int32_t* out_status, float* out_cutoff, int32_t* out_kept,
                         int32_t* out_rounds, void* stream);

/*
 * tps_spec_accept -- speculative acceptance of one draft token per row on truncated distributions
 * ("Top-p (Nucleus) Sampling, in depth", 'Logprobs, speculative decoding and reproducibility': accept
 * a draft token x with probability min(1, P(x)/Q(x)); on rejection draw from the normalised positive
 * part of P - Q, which reproduces P exactly; P is the target's truncated and renormalised
 * distribution, Q the one the draft actually sampled from, truncation included).
 *
 *   P, Q    the renormalised kept distributions tps_sample draws from, for the target row under
 *           (target_temperature, target_top_k, target_top_p, target_min_p) and for the draft row
 *           under the draft's four parameters (one-hot for a greedy row).
 *   The row accepts x iff u Q(x) < P(x) (u: the acceptance uniform); otherwise its token is the
 *   argmax over i with r_i = P(i) - Q(i) > 0 of ln r_i - ln(-ln u_i), lowest index on equal keys.
 *   Uniforms: u = (2 (w >> 9) + 1) 2^-24 with w = word (i mod 4) of Philox4x32-10, key = seed[b] and
 *   counter (i / 4, b | 2^31, step low word, step high word); i = 2^20 - 1 gives the acceptance
 *   uniform.  (Bit 31 of the row word keeps these apart from the sampling draw's counters.)
 *
 *   target_logits, draft_logits  [B, ld] of the same dtype (TPS_F32 / TPS_BF16), V <= ld.
 *   draft_token  [B] int32: the token the draft model drew for the row.
 *   seed         [B] uint64;  step: 64-bit counter word, as in tps_sample.
 *   out_token    [B] int32: x if accepted, else the residual draw; -1 for a failed row.
 *   out_accepted [B] int32 or NULL: 1 if x was accepted, else 0 (0 for a failed row).
 *   out_status   [B] int32 or NULL: a tps_row_status -- the target row's failure first, then the
 *                draft row's; TPS_ROW_BAD_PARAM also when x is outside [0, V) or Q(x) = 0 (the draft
 *                could not have drawn it).
 * A sequence of k draft tokens is k rows; the caller keeps the tokens up to the first rejection.
 * All pointers are caller-owned device memory; the call allocates nothing and is stream-ordered on
 * `stream`.  Returns TPS_ERR_ARG / _DTYPE / _ALIGN / _UNSUPPORTED_V / _CUDA as tps_sample does.
 */
int tps_spec_accept(const void* target_logits, const void* draft_logits, int dtype, int64_t B, int64_t V, int64_t ld,
                    const float* target_temperature, const int32_t* target_top_k, const float* target_top_p,
                    const float* target_min_p, const float* draft_temperature, const int32_t* draft_top_k,
                    const float* draft_top_p, const float* draft_min_p, const int32_t* draft_token,
                    const uint64_t* seed, uint64_t step, int32_t* out_token, int32_t* out_accepted,
                    int32_t* out_status, void* stream);

/*
 * tps_sample_noalloc -- tps_sample_full for callers that cannot allocate device memory while they
 * sample (a serving loop that reserves all device memory up front, a host whose allocator belongs to
 * another framework, code that must stay out of the driver's allocator).  The pages define no such
 * call; it is this library's own.  Same arguments, rules and results as tps_sample_full; the only
 * difference is where the streaming kernel's small per-call scratch lives: tps_sample_full draws it
 * from a stream-ordered memory pool the library keeps per device, this call uses a fixed array of
 * 8 MiB compiled into the library (held on every GPU that loads the library until the process exits)
 * and allocates nothing.
 *   - A call whose scratch would exceed 8 MiB returns TPS_ERR_SCRATCH before enqueuing anything.
 *     The scratch holds 4 bytes per row plus, for a batch of fewer than four rows per SM, about
 *     2 KB per segment of its split rows (at most about 2.5 MB): only batches of about two million
 *     rows or more exceed it.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress): make
 *     that first call before any stream capture.
 *   - Every call shares the one array and clears the part that must start at zero itself, on its
 *     stream.  Calls that overlap on the GPU race on the array: issue them in one stream, or order
 *     their streams.
 */
int tps_sample_noalloc(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld, const float* temperature,
                       const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                       uint64_t step, int32_t* out_token, float* out_probs, int32_t* out_status, float* out_cutoff,
                       int32_t* out_kept, float* out_logprob, int32_t n_top, int32_t* out_top_idx,
                       float* out_top_logprob, int kernel, void* stream);

/*
 * tps_sample_stall_test -- a test hook for the bounded waits (not for production use).  Samples like
 * tps_sample_ex with the streaming kernel, except that CTA 0 withholds the copy of its chunk number
 * `stall_chunk` (counted from 0; -1: none), so that stage never fills, and every wait for data or
 * for a hand-over gives up after `wait_ns` nanoseconds (1 .. 10^9) instead of one second.  The
 * waits for copies already in flight keep their full limit.  Rows the stalled CTA could not finish
 * report TPS_ROW_TIMEOUT with token -1; every other row is sampled as usual; the call returns and
 * the context stays usable.  Returns TPS_ERR_ARG for wait_ns outside that range.
 */
int tps_sample_stall_test(const void* logits, int dtype, int64_t B, int64_t V, const float* temperature,
                          const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seed,
                          uint64_t step, int32_t* out_token, int32_t* out_status, int64_t stall_chunk,
                          uint64_t wait_ns, void* stream);

/* Kernels one tps_sample_kernel call with these arguments launches (0 for arguments the call would
 * reject): 1 for the cluster kernel alone; 2 for the streaming kernel (a one-CTA kernel clears its
 * scratch first); 3 for a split batch (those two, then the cluster kernel).  Host-only query. */
int tps_kernels_per_call(int dtype, int64_t B, int64_t V, int kernel);

/* Largest V the library accepts for `dtype` on the current device (0 for an unknown dtype or
 * when no device is usable); the exact 64-bit mass sums bound it at 2^20 - 1.  Host-only query;
 * enqueues nothing. */
int64_t tps_max_vocab(int dtype);

/* Cluster size (CTAs per row) the cluster kernel would use for this shape on the current device,
 * or 0 when 16 CTAs cannot hold the row.  Host-only query. */
int tps_cluster_size(int dtype, int64_t B, int64_t V);

/* Static, human-readable text for a tps_status or (offset by 100) a tps_row_status. */
const char* tps_status_string(int status);

/* The last cudaError_t seen by a call that returned TPS_ERR_CUDA on this host thread. */
int tps_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int tps_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TPS_H_ */
