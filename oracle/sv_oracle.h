/*
 * sv_oracle.h -- declarations of the float64 CPU oracle for speculative-decoding
 * verification.
 *
 * TEST INFRASTRUCTURE ONLY. The oracle is the slow, plain, obviously-correct
 * statement of what the verification step computes. Only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg load it. The CUDA library
 * never includes, links or calls anything declared here, and this header shares
 * nothing with the library's own header.
 *
 * Conventions (fixed by the pages, see sv_oracle.c for the citations):
 *   p = target distribution, q = draft distribution, both softmax(logits / T).
 *   target rows: [B, K+1, V]; row i < K verifies draft token x_i, row K is the
 *   bonus row. draft rows: [B, K, V]. Row-major, contiguous.
 *   dtype 0 = IEEE binary32, dtype 1 = bfloat16 (raw 16-bit patterns),
 *   dtype 2 = IEEE binary64 (logits an LM head computed exactly, e.g. from
 *   bfloat16 hidden states and weights).
 */
#ifndef SV_ORACLE_H
#define SV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { SVO_F32 = 0, SVO_BF16 = 1, SVO_F64 = 2 };
enum { SVO_SAMPLE = 0, SVO_GREEDY = 1 };

/* Per-sequence status bits written by svo_verify. */
enum { SVO_BAD_TOKEN = 1, SVO_NONFINITE = 2 };

/* Philox4x32 with 10 rounds, one block: out = Philox(ctr, key). */
void svo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* svo_philox4x32_10 for n counters: ctr and out are [n][4]. */
void svo_philox_many(const uint32_t* ctr, int64_t n, const uint32_t key[2], uint32_t* out);

/* Uniform in [0, 1 - 2^-24] from lane `lane` (0..3) of Philox4x32-10 with
 * key = (lo32(seed), hi32(seed)) and counter = (pos, seq, 0, 0). */
double svo_uniform(uint64_t seed, uint32_t seq, uint32_t pos, int lane);

/* Value of element k of a row, exactly widened to double. */
double svo_elem(const void* row, int64_t k, int dtype);

/* Natural-log log-sum-exp of the row scaled by 1/T. Returns 0 on success, or
 * SVO_NONFINITE (and *lse = NaN) when the row holds a NaN or +inf, or is all -inf. */
int svo_row_lse(const void* row, int64_t V, int dtype, double T, double* lse);

/* log p(k) = l_k / T - lse for one row. */
double svo_log_prob(const void* row, int64_t k, int dtype, double T, double lse);

/* Acceptance probability min(1, p/q) from the two log-probabilities. */
double svo_accept_prob(double log_p, double log_q);

/* Sampling weights: w_k = max(0, p_k - q_k) when draft_row != NULL (residual
 * after a rejection), else w_k = p_k (bonus row). */
void svo_sample_weights(const void* target_row, const void* draft_row, int64_t V, int dtype,
                        double T, double lse_t, double lse_d, double* w);

/* Race uniform of token k at emitted position `pos` of sequence `seq`: lane
 * k mod 4 of Philox4x32-10 with key (lo32(seed), hi32(seed)) and counter
 * (pos, seq, 1 + k div 4, 0), mapped to (2 (word >> 9) + 1) * 2^-24 in (0, 1). */
double svo_race_uniform(uint64_t seed, uint32_t seq, uint32_t pos, uint32_t k);

/* Race uniform of block c: as above with counter (pos, seq, 1 + c div 4, 1). */
double svo_block_uniform(uint64_t seed, uint32_t seq, uint32_t pos, uint32_t c);

/* Two-level exponential race over blocks of `block` consecutive tokens (the
 * last block may be shorter): the block with the largest W_c / E_c (W_c = sum
 * of w over the block), then the token of that block with the largest
 * w_k / E_k, E = -ln(uniform). The lowest index wins exact ties. *margin gets
 * the smaller of the two levels' relative gaps (best - second) / best (1 when
 * a level has one candidate, 0 when no weight is positive). Returns -1 if no
 * weight is positive or block < 1.
 *
 * The draw follows w / Z for every block length: level 1 picks block c with
 * probability W_c / Z and level 2 token k of it with probability w_k / W_c,
 * from disjoint clocks. With block >= V there is one block, and the draw is
 * the plain one-level race argmax_k w_k / E_k over the per-token clocks. The
 * length only decides which random numbers are used, so it is a parameter of
 * the reading, passed in by the caller. */
int64_t svo_race_sample(const double* w, int64_t V, int64_t block, uint64_t seed, uint32_t seq,
                        uint32_t pos, double* margin);

/* Lowest index attaining the maximum of the raw row; *has_nan set to 1 when the
 * row holds a NaN (the index is then meaningless). */
int64_t svo_row_argmax(const void* row, int64_t V, int dtype, int* has_nan);

/*
 * Verify sequences b in [b0, b1) of a batch of B.
 *   target      [B, K+1, V]       draft [B, K, V] (unused, may be NULL, when greedy)
 *   tokens      [B, K] int32 (may be NULL when K == 0)
 *   out_tokens  [B, K+1] int32    num_accepted [B] int32
 * Optional outputs (NULL to skip), all indexed like the inputs:
 *   lse_t [B, K+1], lse_d [B, K], log_ratio [B, K]  (sampling mode only)
 *   accept_margin [B, K]: |u_i - r_i| for every decision taken, NaN elsewhere
 *   sample_margin [B]:    smaller relative gap (best - second) / best of the
 *                         race's two levels (0 when the zero-residual fall-back
 *                         fired; NaN in greedy)
 *   seq_status [B]
 * race_block (>= 1) is the block length of the corrected / bonus token's race
 * (svo_race_sample); the CUDA library draws with 512.
 * Returns 0, or -1 on an invalid argument.
 */
int svo_verify(const void* target, const void* draft, const int32_t* tokens,
               int64_t B, int64_t K, int64_t V, int dtype, double T, uint64_t seed, int mode,
               int64_t race_block, int64_t b0, int64_t b1, int32_t* out_tokens,
               int32_t* num_accepted, double* lse_t, double* lse_d, double* log_ratio,
               double* accept_margin, double* sample_margin, int32_t* seq_status);

/*
 * Top-k / top-p cut of one row (logits of `row` over T, natural-log normaliser
 * lse): *thr = the smallest logit value kept (every token with logit >= *thr
 * is kept), *log_mass = log of the kept softmax mass, *margin = the top-p
 * boundary's distance, relative to the top-k set's mass, between top_p and the
 * masses just above and just including the boundary value (+inf when top-p is
 * off). top_k <= 0 or >= V, and top_p >= 1, switch a cut off. Returns 0.
 */
int svo_filter_row(const void* row, int64_t V, int dtype, double T, double lse, int64_t top_k,
                   double top_p, double* thr, double* log_mass, double* margin);

/*
 * svo_verify with both rows of every position filtered by top-k then top-p
 * before the acceptance test and the residual / bonus draw (greedy mode
 * ignores the filters: they never remove a row's maximum). filter_margin_t
 * [B, K+1] and filter_margin_d [B, K] (optional) get each row's top-p boundary
 * margin; filter_thr and filter_log_mass [B, 2K+1] (optional: target rows 0..K,
 * then draft rows 0..K-1) each row's threshold and log kept mass (-inf and 0
 * without filtering). top_p must lie in (0, 1]. A draft token the filtered
 * target gives probability 0 is rejected.
 */
int svo_verify_filtered(const void* target, const void* draft, const int32_t* tokens,
                        int64_t B, int64_t K, int64_t V, int dtype, double T, uint64_t seed,
                        int mode, int64_t race_block, int64_t top_k, double top_p, int64_t b0,
                        int64_t b1, int32_t* out_tokens, int32_t* num_accepted, double* lse_t,
                        double* lse_d, double* log_ratio, double* accept_margin,
                        double* sample_margin, double* filter_margin_t, double* filter_margin_d,
                        double* filter_thr, double* filter_log_mass, int32_t* seq_status);

#ifdef __cplusplus
}
#endif

#endif /* SV_ORACLE_H */
