/*
 * sv_oracle.c -- float64 CPU oracle for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY. Plain, single-threaded, slow on purpose: every
 * step is written out in the order the pages give it, in double precision,
 * with no fusion or reordering. The one blocked step is the draw of the
 * corrected / bonus token: the pages fix only its law, and it is read here as
 * a two-level race over blocks of tokens whose length is an argument (below).
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load this file's library; the CUDA library shares no code with it and never
 * calls it.
 *
 * Pages this follows (cited by title and section):
 *  [RU] "Как работает speculative decoding на уровне логитов, а не токенов?"
 *       (aivaro.ru): §5 "Алгоритм ... (пошагово)", step 3 (accept when
 *       p_target >= p_draft, else reject with probability 1 - p_target/p_draft;
 *       discard every later draft; resample from max(0, p_target - p_draft)/Z)
 *       and §6 (accept(x) = min(1, p_target(x)/p_draft(x))).
 *  [VN] "Speculative decoding" (aihero.vn): section "Chấp nhận bằng tỉ lệ,
 *       không chỉ bằng argmax" (q = draft, p = target, acceptance
 *       min(1, p(x)/q(x)), residual proportional to max(0, p - q), normalised;
 *       verification stops at the first rejection), the paragraph on
 *       temperature/top-k/top-p (transforms applied consistently to both
 *       distributions), and "Cùng phân bố không có nghĩa cùng chuỗi" (greedy
 *       decoding uses a different check from sampling).
 *  [ZH] Hung-yi Lee, "Introduction to Generative AI 2024 Spring", lecture 16
 *       notes (CSDN): §4 "推测解码验证流程图", item 1 (target distribution P_i
 *       is computed at the position before draft token i), item 3 (truncate at
 *       the failed position, emit the target's own token there) and item 4
 *       "The Bonus Token" (all k accepted => one more token from the next
 *       target distribution).
 *  [PH] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *       1, 2, 3", SC'11, §4: the Philox4x32 bijection and its key schedule.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - temperature divides both logit rows before the softmax; greedy ignores it;
 *  - target row i verifies draft token x_i; target row K is the bonus row;
 *  - accept iff u < r with u drawn in [0, 1) (the pseudocode's strict test);
 *  - u_i = lane 0 of Philox(key = seed, counter = (i, b, 0, 0)), mapped to
 *    (32-bit word >> 8) * 2^-24, exact in float and double;
 *  - the pages draw the corrected token with a generic multinomial draw; it is
 *    read here as a two-level exponential race over blocks of L consecutive
 *    tokens, L an argument of the verifier (the CUDA library uses L = 512, a
 *    length picked for its kernels; the law below holds for every L, and
 *    L >= V is the plain one-level race over per-token clocks).
 *    Level 1 races the blocks: block c = argmax over blocks with W_c > 0 of
 *    W_c / E_c, W_c the sum of w over the block, E_c = -ln v_c, v_c lane c mod 4
 *    of counter (j, b, 1 + c div 4, 1). Level 2 races the tokens of the winning
 *    block: token = argmax over its k with w_k > 0 of w_k / E_k, E_k = -ln v_k,
 *    v_k lane k mod 4 of counter (j, b, 1 + k div 4, 0). Uniforms are
 *    (2 (word >> 9) + 1) * 2^-24 in (0, 1); the lowest index wins an exact tie.
 *    The first arrival of independent exponential clocks with rates w_k is
 *    clock k with probability w_k / sum(w), so block c wins with probability
 *    W_c / Z and token k of it with probability w_k / W_c: a draw from w / Z;
 *  - if every residual weight rounds to 0 (possible only through rounding),
 *    p_j is raced instead;
 *  - greedy: lowest index attaining the maximum raw logit; accept while it
 *    equals the draft token; emit the target's argmax at the first mismatch,
 *    or the bonus row's argmax when all K match;
 *  - positions after the emitted token are -1;
 *  - a row holding NaN or +inf, or all -inf, makes the sequence invalid in
 *    sampling mode; a NaN in a target row does so in greedy mode; a draft token
 *    outside [0, V) does so in both modes. Invalid sequences report
 *    num_accepted = -1, all out_tokens = -1 and a status bit.
 */
#include "sv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 [PH] §4.                                                     */
/* One round: two 32x32->64 multiplications of words 0 and 2 by the round     */
/* multipliers; the high halves are xored with the other two words and the    */
/* round key, and the words are permuted. The key is bumped by the Weyl        */
/* constants (golden ratio and sqrt(3) - 1, as 32-bit fractions) each round.  */
/* ------------------------------------------------------------------------- */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void svo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    int round;
    for (round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

void svo_philox_many(const uint32_t* ctr, int64_t n, const uint32_t key[2], uint32_t* out)
{
    int64_t i;
    for (i = 0; i < n; ++i) svo_philox4x32_10(ctr + 4 * i, key, out + 4 * i);
}

double svo_uniform(uint64_t seed, uint32_t seq, uint32_t pos, int lane)
{
    uint32_t ctr[4], key[2], r[4];
    ctr[0] = pos; ctr[1] = seq; ctr[2] = 0; ctr[3] = 0;
    key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    key[1] = (uint32_t)(seed >> 32);
    svo_philox4x32_10(ctr, key, r);
    return (double)(r[lane & 3] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------- */
/* Element access. bfloat16 is the upper half of an IEEE binary32, so placing */
/* its 16 bits in the high half of a 32-bit word gives the float exactly.     */
/* ------------------------------------------------------------------------- */
double svo_elem(const void* row, int64_t k, int dtype)
{
    float f;
    if (dtype == SVO_F64) {
        double d;
        memcpy(&d, (const unsigned char*)row + 8 * k, 8);
        return d;
    }
    if (dtype == SVO_F32) {
        memcpy(&f, (const unsigned char*)row + 4 * k, 4);
    } else {
        uint16_t h;
        uint32_t bits;
        memcpy(&h, (const unsigned char*)row + 2 * k, 2);
        bits = (uint32_t)h << 16;
        memcpy(&f, &bits, 4);
    }
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Softmax of logits / T, through its log-normaliser ([RU] §9 applies a       */
/* softmax to each row; [VN] asks for the temperature on both rows).          */
/* lse = m + log(sum_k exp(s_k - m)), s_k = l_k / T, m = max_k s_k.           */
/* ------------------------------------------------------------------------- */
int svo_row_lse(const void* row, int64_t V, int dtype, double T, double* lse)
{
    double m = -INFINITY, acc = 0.0;
    int64_t k;
    for (k = 0; k < V; ++k) {
        double s = svo_elem(row, k, dtype) / T;
        if (isnan(s) || s == INFINITY) {
            *lse = NAN;
            return SVO_NONFINITE;
        }
        if (s > m) m = s;
    }
    if (m == -INFINITY) {
        *lse = NAN;
        return SVO_NONFINITE;
    }
    for (k = 0; k < V; ++k) acc += exp(svo_elem(row, k, dtype) / T - m);
    *lse = m + log(acc);
    return 0;
}

double svo_log_prob(const void* row, int64_t k, int dtype, double T, double lse)
{
    return svo_elem(row, k, dtype) / T - lse;
}

/* [RU] §6, [VN]: accept(x) = min(1, p(x)/q(x)), taken in the log domain so     */
/* that q(x) underflowing to 0 still gives ratio +inf, i.e. 1.                 */
double svo_accept_prob(double log_p, double log_q)
{
    if (log_p >= log_q) return 1.0;
    return exp(log_p - log_q);
}

/* log p'(x) of a filtered row: -inf below the threshold. */
static double filtered_log_prob(const void* row, int64_t k, int dtype, double T, double lse,
                                double thr, double log_mass)
{
    if (!(svo_elem(row, k, dtype) >= thr)) return -INFINITY;
    return svo_log_prob(row, k, dtype, T, lse) - log_mass;
}

/* [RU] §5 step 3 / §6 and [VN]: after a rejection the next token comes from    */
/* max(0, p - q)/Z; [ZH] §4 item 4: after K acceptances it comes from the       */
/* bonus row's own distribution p. Written for the filtered rows p' and q'    */
/* (threshold -inf and log mass 0: no filter); draft_row NULL gives p'.        */
static void filtered_weights(const void* trow, const void* drow, int64_t V, int dtype, double T,
                             double lse_t, double thr_t, double lm_t, double lse_d, double thr_d,
                             double lm_d, double* w)
{
    int64_t k;
    for (k = 0; k < V; ++k) {
        double p = exp(filtered_log_prob(trow, k, dtype, T, lse_t, thr_t, lm_t));
        if (drow != NULL) {
            double q = exp(filtered_log_prob(drow, k, dtype, T, lse_d, thr_d, lm_d));
            w[k] = (p > q) ? (p - q) : 0.0;
        } else {
            w[k] = p;
        }
    }
}

void svo_sample_weights(const void* target_row, const void* draft_row, int64_t V, int dtype,
                        double T, double lse_t, double lse_d, double* w)
{
    filtered_weights(target_row, draft_row, V, dtype, T, lse_t, -INFINITY, 0.0, lse_d, -INFINITY,
                     0.0, w);
}

/* ------------------------------------------------------------------------- */
/* Top-k / top-p ([VN], paragraph on temperature, top-k and top-p: whatever    */
/* transform the draft's distribution gets, the target's gets the same). Read  */
/* here, for one row, as: keep the tokens whose logit is >= the k-th largest   */
/* logit (every tie at the boundary kept); among those, with their softmax     */
/* renormalised over them, keep the tokens whose logit is >= the largest value */
/* v such that the kept tokens with logit >= v hold at least top_p of the      */
/* mass. Both cuts are a threshold on the logit value, so equal logits are     */
/* kept or dropped together. top_k <= 0 or >= V and top_p >= 1 switch a cut   */
/* off. The filtered distribution is p' = p [logit >= thr] / M.               */
/* ------------------------------------------------------------------------- */
static int cmp_desc(const void* a, const void* b)
{
    double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

int svo_filter_row(const void* row, int64_t V, int dtype, double T, double lse, int64_t top_k,
                   double top_p, double* thr, double* log_mass, double* margin)
{
    double* v = (double*)malloc(sizeof(double) * (size_t)V);
    double thr_k = -INFINITY, mass_k = 0.0, kept = 0.0;
    int64_t k, g;
    if (v == NULL) return -1;
    for (k = 0; k < V; ++k) v[k] = svo_elem(row, k, dtype);
    qsort(v, (size_t)V, sizeof(double), cmp_desc);
    if (top_k > 0 && top_k < V) thr_k = v[top_k - 1];
    for (k = 0; k < V && v[k] >= thr_k; ++k) mass_k += exp(v[k] / T - lse);
    *thr = thr_k;
    *margin = INFINITY;
    if (top_p < 1.0) {
        /* Walk the groups of equal logits from the largest down. */
        const double target = top_p * mass_k;
        double before = 0.0;
        for (k = 0; k < V && v[k] >= thr_k; k = g) {
            double group = 0.0, after;
            for (g = k; g < V && v[g] == v[k]; ++g) group += exp(v[g] / T - lse);
            after = before + group;
            if (after >= target) {
                double m1 = (after - target) / mass_k, m2 = (target - before) / mass_k;
                *thr = v[k] > thr_k ? v[k] : thr_k;
                *margin = m1 < m2 ? m1 : m2;
                break;
            }
            before = after;
        }
    }
    for (k = 0; k < V && v[k] >= *thr; ++k) kept += exp(v[k] / T - lse);
    *log_mass = log(kept);
    free(v);
    return 0;
}

double svo_race_uniform(uint64_t seed, uint32_t seq, uint32_t pos, uint32_t k)
{
    uint32_t ctr[4], key[2], r[4];
    ctr[0] = pos; ctr[1] = seq; ctr[2] = 1u + (k >> 2); ctr[3] = 0;
    key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    key[1] = (uint32_t)(seed >> 32);
    svo_philox4x32_10(ctr, key, r);
    return (double)(2u * (r[k & 3u] >> 9) + 1u) * (1.0 / 16777216.0);
}

double svo_block_uniform(uint64_t seed, uint32_t seq, uint32_t pos, uint32_t c)
{
    uint32_t ctr[4], key[2], r[4];
    ctr[0] = pos; ctr[1] = seq; ctr[2] = 1u + (c >> 2); ctr[3] = 1;
    key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    key[1] = (uint32_t)(seed >> 32);
    svo_philox4x32_10(ctr, key, r);
    return (double)(2u * (r[c & 3u] >> 9) + 1u) * (1.0 / 16777216.0);
}

/* One exponential race: keep the largest w / E and the second largest. */
static void race_step(double w, double v, int64_t id, double* best, double* second, int64_t* best_id)
{
    double score = w / (-log(v));
    if (score > *best) {
        if (*best_id >= 0) *second = *best;
        *best = score;
        *best_id = id;
    } else if (score > *second) {
        *second = score;
    }
}

int64_t svo_race_sample(const double* w, int64_t V, int64_t block, uint64_t seed, uint32_t seq,
                        uint32_t pos, double* margin)
{
    double best = -INFINITY, second = 0.0, gap1, gap2;
    int64_t nblocks, c, k, best_c = -1, best_k = -1, k0, k1;
    if (block < 1) {
        *margin = 0.0;
        return -1;
    }
    nblocks = (V + block - 1) / block;
    /* Level 1: the blocks, each with the total weight of its tokens. */
    for (c = 0; c < nblocks; ++c) {
        double W = 0.0;
        k0 = c * block;
        k1 = k0 + block < V ? k0 + block : V;
        for (k = k0; k < k1; ++k) W += w[k];
        if (W > 0.0) race_step(W, svo_block_uniform(seed, seq, pos, (uint32_t)c), c, &best, &second, &best_c);
    }
    if (best_c < 0) {
        *margin = 0.0;
        return -1;
    }
    gap1 = (best - second) / best;
    /* Level 2: the tokens of the winning block. */
    best = -INFINITY;
    second = 0.0;
    k0 = best_c * block;
    k1 = k0 + block < V ? k0 + block : V;
    for (k = k0; k < k1; ++k)
        if (w[k] > 0.0) race_step(w[k], svo_race_uniform(seed, seq, pos, (uint32_t)k), k, &best, &second, &best_k);
    gap2 = (best - second) / best;
    *margin = gap1 < gap2 ? gap1 : gap2;
    return best_k;
}

/* Greedy check ([VN], "Cùng phân bố..."): the raw-logit argmax; the lowest     */
/* index wins ties.                                                              */
int64_t svo_row_argmax(const void* row, int64_t V, int dtype, int* has_nan)
{
    int64_t k, best_k = 0;
    double best = -INFINITY;
    *has_nan = 0;
    for (k = 0; k < V; ++k) {
        double v = svo_elem(row, k, dtype);
        if (isnan(v)) *has_nan = 1;
        else if (v > best) {
            best = v;
            best_k = k;
        }
    }
    return best_k;
}

/* ------------------------------------------------------------------------- */
/* One sequence.                                                              */
/* ------------------------------------------------------------------------- */
static void fail_sequence(int64_t b, int64_t K, int32_t status, int32_t* out_tokens,
                          int32_t* num_accepted, int32_t* seq_status)
{
    int64_t i;
    for (i = 0; i <= K; ++i) out_tokens[b * (K + 1) + i] = -1;
    num_accepted[b] = -1;
    if (seq_status) seq_status[b] = status;
}

static void verify_sampling(const void* target, const void* draft, const int32_t* tokens,
                            int64_t b, int64_t K, int64_t V, int dtype, double T, uint64_t seed,
                            int64_t race_block, int64_t top_k, double top_p, int32_t* out_tokens,
                            int32_t* num_accepted, double* lse_t_out, double* lse_d_out,
                            double* log_ratio_out, double* accept_margin, double* sample_margin,
                            double* fm_t, double* fm_d, double* thr_out, double* lm_out,
                            int32_t* seq_status)
{
    const int filtering = (top_k > 0 && top_k < V) || top_p < 1.0;
    const size_t esz = (dtype == SVO_F64) ? 8 : (dtype == SVO_F32) ? 4 : 2;
    const unsigned char* trow0 = (const unsigned char*)target + (size_t)(b * (K + 1)) * V * esz;
    const unsigned char* drow0 =
        draft ? (const unsigned char*)draft + (size_t)(b * K) * V * esz : NULL;
    double* lse_t = (double*)malloc(sizeof(double) * (size_t)(K + 1));
    double* lse_d = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    /* Thresholds and log kept masses of the filtered rows: [0, K] target, then
     * [K + 1, 2K] draft (no filtering: -inf and 0). */
    double* thr = (double*)malloc(sizeof(double) * (size_t)(2 * K + 1));
    double* lm = (double*)malloc(sizeof(double) * (size_t)(2 * K + 1));
    int32_t status = 0;
    int64_t i, j;
    double margin;
    int64_t token;

    /* Every draft token must name a vocabulary entry. */
    for (i = 0; i < K; ++i) {
        int32_t x = tokens[b * K + i];
        if (x < 0 || (int64_t)x >= V) status |= SVO_BAD_TOKEN;
    }
    /* Step 1: the normaliser of every target row (K verify rows + bonus row)   */
    /* and every draft row.                                                     */
    for (i = 0; i <= K; ++i)
        status |= svo_row_lse(trow0 + (size_t)i * V * esz, V, dtype, T, &lse_t[i]);
    for (i = 0; i < K; ++i)
        status |= svo_row_lse(drow0 + (size_t)i * V * esz, V, dtype, T, &lse_d[i]);
    for (i = 0; i <= K; ++i)
        if (lse_t_out) lse_t_out[b * (K + 1) + i] = lse_t[i];
    for (i = 0; i < K; ++i)
        if (lse_d_out) lse_d_out[b * K + i] = lse_d[i];
    if (accept_margin)
        for (i = 0; i < K; ++i) accept_margin[b * K + i] = NAN;
    if (sample_margin) sample_margin[b] = NAN;
    for (i = 0; i <= 2 * K; ++i) {
        thr[i] = -INFINITY;
        lm[i] = 0.0;
    }
    if (fm_t)
        for (i = 0; i <= K; ++i) fm_t[b * (K + 1) + i] = INFINITY;
    if (fm_d)
        for (i = 0; i < K; ++i) fm_d[b * K + i] = INFINITY;
    if (status != 0) {
        fail_sequence(b, K, status, out_tokens, num_accepted, seq_status);
        goto done;
    }
    if (filtering) {
        double mg;
        for (i = 0; i <= K; ++i) {
            svo_filter_row(trow0 + (size_t)i * V * esz, V, dtype, T, lse_t[i], top_k, top_p,
                           &thr[i], &lm[i], &mg);
            if (fm_t) fm_t[b * (K + 1) + i] = mg;
        }
        for (i = 0; i < K; ++i) {
            svo_filter_row(drow0 + (size_t)i * V * esz, V, dtype, T, lse_d[i], top_k, top_p,
                           &thr[K + 1 + i], &lm[K + 1 + i], &mg);
            if (fm_d) fm_d[b * K + i] = mg;
        }
    }
    /* Thresholds and log kept masses, [B][2K + 1] (target rows, then draft). */
    if (thr_out)
        for (i = 0; i <= 2 * K; ++i) thr_out[b * (2 * K + 1) + i] = thr[i];
    if (lm_out)
        for (i = 0; i <= 2 * K; ++i) lm_out[b * (2 * K + 1) + i] = lm[i];

    /* Log ratio log p_i(x_i) - log q_i(x_i) at every position (diagnostic). */
    for (i = 0; i < K; ++i) {
        int32_t x = tokens[b * K + i];
        double lp = filtered_log_prob(trow0 + (size_t)i * V * esz, x, dtype, T, lse_t[i], thr[i],
                                      lm[i]);
        double lq = filtered_log_prob(drow0 + (size_t)i * V * esz, x, dtype, T, lse_d[i],
                                      thr[K + 1 + i], lm[K + 1 + i]);
        if (log_ratio_out) log_ratio_out[b * K + i] = lp - lq;
    }

    /* Step 2: positions in order; accept x_i with probability min(1, p/q);     */
    /* the first rejection ends the scan ([RU] §5 step 3, [VN], [ZH] §4 item 3). */
    j = K;
    for (i = 0; i < K; ++i) {
        int32_t x = tokens[b * K + i];
        double lp = filtered_log_prob(trow0 + (size_t)i * V * esz, x, dtype, T, lse_t[i], thr[i],
                                      lm[i]);
        double lq = filtered_log_prob(drow0 + (size_t)i * V * esz, x, dtype, T, lse_d[i],
                                      thr[K + 1 + i], lm[K + 1 + i]);
        /* A token the filtered target cannot produce is rejected (even when */
        /* the filtered draft cannot produce it either).                      */
        double r = lp == -INFINITY ? 0.0 : svo_accept_prob(lp, lq);
        double u = svo_uniform(seed, (uint32_t)b, (uint32_t)i, 0);
        if (accept_margin) accept_margin[b * K + i] = fabs(u - r);
        if (!(u < r)) {
            j = i;
            break;
        }
    }

    /* Step 3: the token at position j -- the residual after a rejection, the   */
    /* bonus row after K acceptances.                                           */
    if (j < K) {
        filtered_weights(trow0 + (size_t)j * V * esz, drow0 + (size_t)j * V * esz, V, dtype, T,
                         lse_t[j], thr[j], lm[j], lse_d[j], thr[K + 1 + j], lm[K + 1 + j], w);
    } else {
        filtered_weights(trow0 + (size_t)K * V * esz, NULL, V, dtype, T, lse_t[K], thr[K], lm[K],
                         0.0, 0.0, 0.0, w);
    }
    token = svo_race_sample(w, V, race_block, seed, (uint32_t)b, (uint32_t)j, &margin);
    if (token < 0) {
        /* Every residual weight rounded to zero: race p'_j instead. */
        filtered_weights(trow0 + (size_t)j * V * esz, NULL, V, dtype, T, lse_t[j], thr[j], lm[j],
                         0.0, 0.0, 0.0, w);
        token = svo_race_sample(w, V, race_block, seed, (uint32_t)b, (uint32_t)j, &margin);
        margin = 0.0;
    }
    if (sample_margin) sample_margin[b] = margin;

    for (i = 0; i < j; ++i) out_tokens[b * (K + 1) + i] = tokens[b * K + i];
    out_tokens[b * (K + 1) + j] = (int32_t)token;
    for (i = j + 1; i <= K; ++i) out_tokens[b * (K + 1) + i] = -1;
    num_accepted[b] = (int32_t)j;
    if (seq_status) seq_status[b] = 0;

done:
    free(lse_t);
    free(lse_d);
    free(w);
    free(thr);
    free(lm);
}

static void verify_greedy(const void* target, const int32_t* tokens, int64_t b, int64_t K,
                          int64_t V, int dtype, int32_t* out_tokens, int32_t* num_accepted,
                          double* accept_margin, double* sample_margin, int32_t* seq_status)
{
    const size_t esz = (dtype == SVO_F64) ? 8 : (dtype == SVO_F32) ? 4 : 2;
    const unsigned char* trow0 = (const unsigned char*)target + (size_t)(b * (K + 1)) * V * esz;
    int64_t* a = (int64_t*)malloc(sizeof(int64_t) * (size_t)(K + 1));
    int32_t status = 0;
    int64_t i, j;

    for (i = 0; i < K; ++i) {
        int32_t x = tokens[b * K + i];
        if (x < 0 || (int64_t)x >= V) status |= SVO_BAD_TOKEN;
    }
    for (i = 0; i <= K; ++i) {
        int has_nan;
        a[i] = svo_row_argmax(trow0 + (size_t)i * V * esz, V, dtype, &has_nan);
        if (has_nan) status |= SVO_NONFINITE;
    }
    if (accept_margin)
        for (i = 0; i < K; ++i) accept_margin[b * K + i] = NAN;
    if (sample_margin) sample_margin[b] = NAN;
    if (status != 0) {
        fail_sequence(b, K, status, out_tokens, num_accepted, seq_status);
        free(a);
        return;
    }
    j = K;
    for (i = 0; i < K; ++i) {
        if (a[i] != (int64_t)tokens[b * K + i]) {
            j = i;
            break;
        }
    }
    for (i = 0; i < j; ++i) out_tokens[b * (K + 1) + i] = tokens[b * K + i];
    out_tokens[b * (K + 1) + j] = (int32_t)a[j];
    for (i = j + 1; i <= K; ++i) out_tokens[b * (K + 1) + i] = -1;
    num_accepted[b] = (int32_t)j;
    if (seq_status) seq_status[b] = 0;
    free(a);
}

int svo_verify(const void* target, const void* draft, const int32_t* tokens,
               int64_t B, int64_t K, int64_t V, int dtype, double T, uint64_t seed, int mode,
               int64_t race_block, int64_t b0, int64_t b1, int32_t* out_tokens,
               int32_t* num_accepted, double* lse_t, double* lse_d, double* log_ratio,
               double* accept_margin, double* sample_margin, int32_t* seq_status)
{
    return svo_verify_filtered(target, draft, tokens, B, K, V, dtype, T, seed, mode, race_block,
                               0, 1.0, b0, b1, out_tokens, num_accepted, lse_t, lse_d, log_ratio,
                               accept_margin, sample_margin, NULL, NULL, NULL, NULL, seq_status);
}

int svo_verify_filtered(const void* target, const void* draft, const int32_t* tokens,
                        int64_t B, int64_t K, int64_t V, int dtype, double T, uint64_t seed,
                        int mode, int64_t race_block, int64_t top_k, double top_p, int64_t b0,
                        int64_t b1, int32_t* out_tokens, int32_t* num_accepted, double* lse_t,
                        double* lse_d, double* log_ratio, double* accept_margin,
                        double* sample_margin, double* filter_margin_t, double* filter_margin_d,
                        double* filter_thr, double* filter_log_mass, int32_t* seq_status)
{
    int64_t b;
    if (!(top_p > 0.0 && top_p <= 1.0)) return -1;
    if (race_block < 1) return -1;
    if (B < 0 || K < 0 || V < 1 || b0 < 0 || b1 > B || b0 > b1) return -1;
    if (dtype != SVO_F32 && dtype != SVO_BF16 && dtype != SVO_F64) return -1;
    if (mode != SVO_SAMPLE && mode != SVO_GREEDY) return -1;
    if (target == NULL || out_tokens == NULL || num_accepted == NULL) return -1;
    if (K > 0 && tokens == NULL) return -1;
    if (mode == SVO_SAMPLE && (K > 0 && draft == NULL)) return -1;
    if (mode == SVO_SAMPLE && !(T > 0.0 && isfinite(T))) return -1;
    for (b = b0; b < b1; ++b) {
        if (mode == SVO_SAMPLE)
            verify_sampling(target, draft, tokens, b, K, V, dtype, T, seed, race_block, top_k,
                            top_p, out_tokens, num_accepted, lse_t, lse_d, log_ratio, accept_margin,
                            sample_margin, filter_margin_t, filter_margin_d, filter_thr,
                            filter_log_mass, seq_status);
        else
            verify_greedy(target, tokens, b, K, V, dtype, out_tokens, num_accepted,
                          accept_margin, sample_margin, seq_status);
    }
    return 0;
}
