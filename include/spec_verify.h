/*
 * spec_verify.h -- C ABI of libspecverify, batched speculative-decoding
 * verification on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (the pages it follows, by title and section):
 *
 *  - "Как работает speculative decoding на уровне логитов, а не токенов?"
 *    (aivaro.ru) §5 step 3 and §6: for each drafted position, the draft token
 *    x is accepted with probability min(1, p_target(x) / p_draft(x)); at the
 *    first rejection every later draft is dropped and one token is drawn from
 *    max(0, p_target - p_draft) / Z.
 *  - "Speculative decoding" (aihero.vn), section on accepting by ratio:
 *    q is the draft distribution and p the target distribution at the same
 *    prefix; verification stops at the first rejection; temperature (and any
 *    other transform) is applied consistently to both distributions; greedy
 *    decoding uses a different check from sampling.
 *  - Hung-yi Lee, "Introduction to Generative AI 2024 Spring", lecture 16
 *    notes, §4 (verification flowchart), item 4 "The Bonus Token": when all k
 *    drafts pass, the target's distribution at the next position yields one
 *    extra token, so a round emits up to k + 1 tokens.
 *
 * Layout (all row-major and contiguous; b = sequence, i = position):
 *   target_logits [B, K+1, V]  row i < K is the target distribution at the
 *                              position of draft token i; row K is the bonus row.
 *   draft_logits  [B, K, V]    row i produced draft token i.
 *   draft_tokens  [B, K]       int32.
 *   out_tokens    [B, K+1]     int32: x_0 .. x_{j-1}, then the corrected (or
 *                              bonus) token at j, then -1.
 *   num_accepted  [B]          int32: j, the number of drafts kept (0..K);
 *                              -1 when the sequence's inputs are invalid.
 *
 * Numbers and reproducibility:
 *   p = softmax(target_logits / T), q = softmax(draft_logits / T). Sums of
 *   2^(x log2(e) / T) are carried on the device as float pairs (hi + lo)
 *   scaled by integer powers of two; the device path uses no double precision
 *   except to write the optional diagnostic outputs. The acceptance uniform of
 *   position i of sequence b is lane 0 of Philox4x32-10 with key
 *   (lo32(seed), hi32(seed)) and counter (i, b, 0, 0), mapped to
 *   (word >> 8) * 2^-24; position i is kept iff that uniform is below
 *   min(1, p_i(x_i) / q_i(x_i)). The token at the emitted position j is drawn
 *   from the weights w (max(0, p_j - q_j) after a rejection, p_K for the
 *   bonus) by a two-level exponential race over blocks of 512 tokens. Level 1
 *   takes the block c with the largest W_c / E_c over blocks with weight
 *   W_c = sum of w over the block > 0, E_c = -ln v_c, v_c lane (c mod 4) of
 *   counter (j, b, 1 + c div 4, 1). Level 2 takes the token k of that block
 *   with the largest w_k / E_k over w_k > 0, v_k lane (k mod 4) of counter
 *   (j, b, 1 + k div 4, 0). Both levels map a word to (2 (word >> 9) + 1) 2^-24
 *   and let the lowest index win an exact tie. The race picks token k with
 *   probability w_k / sum(w) for any block length; the length (512, so that
 *   one 128-thread block reads a block as one four-token group per thread)
 *   only decides which random numbers the draw uses. Results are a pure
 *   function of (inputs, T, seed, mode) on a given GPU model: no float
 *   atomics, fixed reduction trees, the same answer on every run.
 *
 * Memory and streams:
 *   Every pointer passed to spec_verify / spec_verify_debug / spec_verify_timed
 *   is DEVICE memory owned by the caller. The library allocates nothing and
 *   keeps no state between calls other than a per-device cache of launch
 *   parameters. Calls are asynchronous and stream-ordered: they enqueue work
 *   on `stream` (a cudaStream_t, NULL = legacy default stream) and return
 *   without synchronising. Inputs must stay unchanged, and outputs and
 *   workspace unread, until the stream has passed the call. Two calls that
 *   share a workspace must be ordered on the GPU (same stream or events).
 *
 * Errors:
 *   Functions return SV_OK (0) or a negative SV_ERR_* code. Argument errors
 *   are found on the host before anything is enqueued. Data errors found on
 *   the device (a draft token outside [0, V), a target or draft row holding a
 *   NaN or +inf or made only of -inf in sampling mode, a NaN target row in
 *   greedy mode) make that sequence's num_accepted -1 and its out_tokens all
 *   -1, and set SV_SEQ_* bits in the optional per-sequence status output. No
 *   input, however malformed, makes a kernel read outside the buffers
 *   described here.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Logits storage type. */
enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 };

/* SV_SAMPLE: rejection sampling (acceptance min(1, p/q), residual, bonus).
 * SV_GREEDY: accept while argmax(target row i) == x_i (lowest index wins
 *            ties, raw logits, temperature unused); at the first mismatch,
 *            or at the bonus row, emit the target row's argmax. */
enum sv_mode { SV_SAMPLE = 0, SV_GREEDY = 1 };

enum sv_status {
    SV_OK = 0,
    SV_ERR_ARG = -1,       /* bad size, mode, temperature or NULL pointer   */
    SV_ERR_DTYPE = -2,     /* unknown dtype                                 */
    SV_ERR_ALIGN = -3,     /* logits not 16-byte aligned, ints not 4-byte   */
    SV_ERR_WORKSPACE = -4, /* workspace NULL, too small or not 256-aligned  */
    SV_ERR_CUDA = -5,      /* a CUDA runtime call or launch failed          */
    SV_ERR_SIZE = -6       /* sizes beyond the supported range              */
};

/* Per-sequence status bits (spec_verify_debug's seq_status output). */
enum sv_seq_status {
    SV_SEQ_BAD_TOKEN = 1,  /* a draft token outside [0, V)                  */
    SV_SEQ_NONFINITE = 2,  /* a NaN / +inf / all -inf row (see above)       */
    SV_SEQ_TIMEOUT = 4,    /* a bounded wait inside a kernel expired        */
    SV_SEQ_INDEX = 8       /* a device-side index check failed (the library
                              built with device checks only; see
                              sv_device_checks)                             */
};

/*
 * 1 if this library was built with device-side index checks (the debug
 * variant, libspecverify_debug.so), 0 for the product build. With them every
 * kernel tests the indices it computes or reads before it uses them; a
 * failed test skips that access and reports SV_SEQ_INDEX for the sequence
 * (num_accepted -1, tokens -1), never a trap. Host-only: no CUDA call.
 */
int sv_device_checks(void);

/* Supported ranges: 0 <= B < 2^31, 0 <= K <= 1024, 1 <= V < 2^31,
 * B * (2K + 1) * V * sizeof(element) < 2^62. Temperature (sampling mode):
 * finite, > 0, with log2(e)/T finite in float32. */

/*
 * Workspace needed by spec_verify for these sizes on the CURRENT device.
 * Writes the byte count to *bytes. Returns SV_OK or an SV_ERR_* code.
 */
int sv_workspace_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode, size_t* bytes);

/*
 * Verify B sequences of K drafts each (see the file comment for what that
 * means and for the layouts).
 *   target_logits  device, [B, K+1, V] of `dtype`, 16-byte aligned.
 *   draft_logits   device, [B, K, V] of `dtype`, 16-byte aligned; may be NULL
 *                  when mode == SV_GREEDY or K == 0.
 *   draft_tokens   device, [B, K] int32; may be NULL when K == 0.
 *   temperature    divides both target and draft logits (sampling mode only).
 *   seed           Philox key.
 *   out_tokens     device, [B, K+1] int32, written.
 *   num_accepted   device, [B] int32, written.
 *   workspace      device, >= sv_workspace_bytes(...) bytes, 256-byte aligned,
 *                  any contents; overwritten.
 *   stream         cudaStream_t to enqueue on.
 * B == 0 enqueues nothing and returns SV_OK.
 */
int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                int64_t B, int64_t K, int64_t V, int dtype, float temperature, uint64_t seed,
                int mode, int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                size_t workspace_bytes, void* stream);

/*
 * spec_verify plus the intermediate values the parity tests compare. Same
 * arguments and launches, plus (each device memory, each may be NULL):
 *   lse_t      [B, K+1] double: natural-log log-sum-exp of target_logits / T.
 *   lse_d      [B, K]   double: the same for draft rows.
 *   log_ratio  [B, K]   double: log p_i(x_i) - log q_i(x_i).
 *   seq_status [B]      int32:  SV_SEQ_* bits, 0 for a valid sequence.
 * In greedy mode lse_t / lse_d / log_ratio are not written.
 */
int spec_verify_debug(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                      float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                      int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                      void* stream, double* lse_t, double* lse_d, double* log_ratio,
                      int32_t* seq_status);

/*
 * spec_verify with CUDA events recorded on `stream` between its kernels, for
 * timing the stages in place: events[0] before the row-statistics kernel,
 * events[1] after it, events[2] after the acceptance scan, events[3] after
 * the residual/bonus sampler (equal to events[2]'s position in greedy mode).
 * `events` holds n_events (>= 4) cudaEvent_t handles created by the caller.
 * spec_verify starts each kernel while the previous one drains (programmatic
 * dependent launch); this variant runs them strictly one after another so
 * that the events bracket each stage, so its total can exceed spec_verify's.
 */
int spec_verify_timed(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                      float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                      int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                      void* stream, void* const* events, int n_events);

/*
 * Device staging bytes spec_verify_host needs for these sizes on the current
 * device (inputs + outputs + workspace, each 256-byte aligned).
 */
int sv_host_staging_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode, size_t* bytes);

/*
 * End-to-end call from HOST buffers. Copies target/draft logits and draft
 * tokens from host memory to `staging` (device, >= sv_host_staging_bytes,
 * 256-byte aligned), runs spec_verify on `stream`, and copies out_tokens and
 * num_accepted back to host memory, all enqueued on `stream`. Returns after
 * enqueueing; the host outputs are valid once the stream has been
 * synchronised. Host buffers should be page-locked (cudaHostAlloc) for the
 * copies to be asynchronous; pageable memory works but the copies then
 * synchronise with the host.
 */
int spec_verify_host(const void* h_target_logits, const void* h_draft_logits,
                     const int32_t* h_draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                     float temperature, uint64_t seed, int mode, int32_t* h_out_tokens,
                     int32_t* h_num_accepted, void* staging, size_t staging_bytes, void* stream);

/*
 * spec_verify for callers that cannot allocate device memory. The pages have
 * no counterpart to this entry point; it exists for callers such as code
 * inside a host framework that owns all device memory through its own pool,
 * where a cudaMalloc would fail or break the pool's accounting, or code on a
 * latency-critical path, where cudaMalloc / cudaFree would synchronise the
 * device.
 *
 * Arguments and results are those of spec_verify, without the workspace: the
 * caller still passes its own (device) inputs and outputs. The scratch is a
 * fixed array of 8 MiB inside the library's device image, held by every GPU
 * that loads the library until the process exits. Problems whose
 * sv_workspace_bytes exceed 8 MiB are rejected with SV_ERR_SIZE before
 * anything is enqueued. The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. All calls share the one array: two calls whose
 * work overlaps on the GPU (different streams, no ordering between them) race
 * on it. The array keeps the last call's contents; nothing in it needs to
 * start at zero. The looked-up address is kept for the life of the process:
 * after cudaDeviceReset on a device, unload and reload the library before
 * calling this entry point on that device again.
 */
int spec_verify_static(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                       float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                       int32_t* num_accepted, void* stream);

/*
 * Workspace needed by spec_verify_early_exit for these sizes on the CURRENT
 * device. Writes the byte count to *bytes. Returns SV_OK or an SV_ERR_* code.
 */
int sv_early_exit_workspace_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode,
                                  size_t* bytes);

/*
 * spec_verify that stops reading a sequence's rows at its first rejection
 * (Hung-yi Lee, "Introduction to Generative AI 2024 Spring", lecture 16
 * notes, section on the key engineering optimisations, item 4 "Early Stop":
 * once a draft is found wrong, the later drafts are not verified). The positions are verified in phases of
 * 1, 2, 4, ... positions; each phase reads the target and draft rows of its
 * positions only for the sequences that accepted every earlier draft.
 *
 * Arguments, layouts, results and errors are those of spec_verify, with a
 * workspace of sv_early_exit_workspace_bytes. out_tokens and num_accepted are
 * the same function of the inputs as spec_verify's, with one exception: rows
 * after a sequence's emitted position are never read, so a NaN or +inf there
 * (or a row of only -inf) does not invalidate the sequence. Draft tokens are
 * all checked. The normalisers of a row are merged in another order than in
 * spec_verify, so the two can differ on the decisions the near-tie rule
 * flags (a gap below 1e-5), and only there. Calls make 2 launches per phase
 * (about log2(K + 1) + 1 phases), a small memset, and in sampling mode the two
 * sampler launches.
 */
int spec_verify_early_exit(const void* target_logits, const void* draft_logits,
                           const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                           float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                           int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Workspace needed by spec_verify_sharded for these sizes on the CURRENT
 * device (Vs = columns per shard, G shards). Writes the byte count to *bytes.
 */
int sv_sharded_workspace_bytes(int64_t B, int64_t K, int64_t Vs, int G, int dtype, int mode,
                               size_t* bytes);

/*
 * spec_verify on logits split over the vocabulary, as a tensor-parallel LM
 * head leaves them: shard g holds the columns [g Vs, (g + 1) Vs) of every
 * row. The pages have no counterpart to this entry point; it computes what
 * spec_verify computes on the concatenated logits (the same method, same
 * tokens and counts, same random numbers), on one GPU, without the caller
 * concatenating them. Pass 1 reduces each shard's part of every row, the scan
 * merges the shards' partial normalisers (the exchange a multi-GPU version
 * would make with an allreduce), and the sampler reads each sequence's
 * emitted row pair from the shards (when Vs * sizeof(element) is not a
 * multiple of 16, the pair is first gathered into the workspace).
 *   target_shards  HOST array of G device pointers, shard g: [B, K+1, Vs] of
 *                  `dtype`, 16-byte aligned.
 *   draft_shards   HOST array of G device pointers, shard g: [B, K, Vs]; may
 *                  be NULL when mode == SV_GREEDY or K == 0.
 *   G              1 .. 16.
 *   Vs             columns per shard; V = G Vs, with V < 2^31 (and, for
 *                  G > 1, V at most 65535 * 2048 bf16 or 65535 * 1024 fp32
 *                  columns).
 * Other arguments, outputs and errors as spec_verify; the workspace is
 * sv_sharded_workspace_bytes (with unaligned shard widths in sampling mode it
 * includes a [B][2][V] buffer for the gathered row pairs). The normalisers
 * are merged in another order than spec_verify's, so the two can differ only
 * on decisions the near-tie rule flags.
 */
int spec_verify_sharded(const void* const* target_shards, const void* const* draft_shards, int G,
                        const int32_t* draft_tokens, int64_t B, int64_t K, int64_t Vs, int dtype,
                        float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                        int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * Workspace needed by spec_verify_filtered for these sizes on the CURRENT
 * device. Writes the byte count to *bytes.
 */
int sv_filtered_workspace_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode,
                                size_t* bytes);

/*
 * spec_verify with top-k / top-p applied to both distributions of every
 * position ("Speculative decoding" (aihero.vn), the paragraph on
 * temperature, top-k and top-p: the draft and the target get the same
 * transform). Each row's softmax at `temperature` is cut to the tokens whose
 * logit is >= a threshold and renormalised over them:
 *   top-k  keep the logits >= the top_k-th largest (ties at the boundary are
 *          kept); top_k = 0 or top_k >= V: no top-k cut;
 *   top-p  inside the top-k set, keep the logits >= the largest value v whose
 *          upper set {x >= v} holds at least top_p of the set's mass;
 *          top_p = 1: no top-p cut.
 * The filtered rows p' and q' then replace p and q everywhere: acceptance
 * min(1, p'(x)/q'(x)) (a draft token with p'(x) = 0 is rejected), the
 * residual max(0, p' - q'), the bonus draw from p'_K. Draft tokens should be
 * drawn from q' for the output to follow p'.
 *   top_k   >= 0 (SV_ERR_ARG otherwise).
 *   top_p   in (0, 1] (SV_ERR_ARG otherwise, NaN included).
 * Other arguments, outputs and errors as spec_verify; the workspace is
 * sv_filtered_workspace_bytes. Greedy mode ignores both cuts (they never
 * remove a row's maximum), and with both cuts off the call is spec_verify.
 * Thresholds are exact (integer work on the logits' order); the top-p
 * boundary's masses are 64-bit fixed point, so a boundary that the exact
 * masses put within 1e-5 of top_p (relative to the top-k mass) may fall on
 * the other side. Rows must hold fewer than 2^22 logits (SV_ERR_SIZE
 * otherwise: the 2^40-scaled mass sums of longer rows could overflow 64 bits).
 * Not combined with early exit or sharded logits. Calls make 4 launches:
 * thresholds, scan, and the two sampler launches.
 */
int spec_verify_filtered(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                         float temperature, int64_t top_k, float top_p, uint64_t seed, int mode,
                         int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * spec_verify_filtered plus per-row diagnostics (each output optional, NULL
 * to skip; device memory):
 *   lse_t [B, K+1], lse_d [B, K]  float64, natural-log normaliser of the KEPT
 *                                 tokens: log sum over x >= thr of exp(x / T);
 *   thr_t [B, K+1], thr_d [B, K]  float32, each row's threshold: a token is
 *                                 kept when its logit is >= it (-inf: no cut);
 *   seq_status [B]                int32, SV_SEQ_* bits (0 = valid).
 * Rows of invalid sequences hold unspecified values. lse_* must be 8-byte
 * aligned, the others 4-byte aligned (SV_ERR_ALIGN).
 */
int spec_verify_filtered_debug(const void* target_logits, const void* draft_logits,
                               const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                               int dtype, float temperature, int64_t top_k, float top_p,
                               uint64_t seed, int mode, int32_t* out_tokens,
                               int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                               void* stream, double* lse_t, double* lse_d, float* thr_t,
                               float* thr_d, int32_t* seq_status);

/*
 * spec_verify_filtered with n_events >= 4 cudaEvent_t handles recorded on
 * `stream` before the thresholds launch, after it, after the scan and after
 * the sampler (launches are then not chained programmatically).
 */
int spec_verify_filtered_timed(const void* target_logits, const void* draft_logits,
                               const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                               int dtype, float temperature, int64_t top_k, float top_p,
                               uint64_t seed, int mode, int32_t* out_tokens,
                               int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                               void* stream, void* const* events, int n_events);

/*
 * Workspace needed by spec_verify_lmhead for these sizes on the CURRENT
 * device (d_target / d_draft: hidden sizes). Writes the byte count to *bytes.
 */
int sv_lmhead_workspace_bytes(int64_t B, int64_t K, int64_t V, int64_t d_target,
                              int64_t d_draft, int mode, size_t* bytes);

/*
 * spec_verify from the models' last hidden states instead of their logits.
 * The pages take each model's logits as given: one vector of V logits per
 * position ("Как работает speculative decoding на уровне логитов..."
 * (aivaro.ru) §4 and §5 step 1). A language model makes them with its output
 * layer, logits = h W^T for a hidden state h and an output matrix W [V, D];
 * this entry point computes that product on the tensor cores and folds the
 * row statistics into it, so the [B, 2K+1, V] logits are never written:
 *   1. one GEMM over every target and draft row yields, per 256-column
 *      vocabulary tile, the row's partial softmax normaliser at `temperature`
 *      (greedy: the tile's maximum and its lowest column) and the draft
 *      token's logit;
 *   2. the scan merges the partials and takes the acceptance decisions
 *      exactly as spec_verify does;
 *   3. (sampling) the hidden states of each sequence's emitted position are
 *      gathered and a second GEMM writes that position's target and draft
 *      logits ([B][2][V] float32, in the workspace), from which the sampler
 *      draws the residual or bonus token as spec_verify does.
 *   hidden_target  device, [B, K+1, d_target] bfloat16, row-major, 16-byte
 *                  aligned: the target model's hidden state at every verified
 *                  position (position i < K scores draft token x_i, position
 *                  K is the bonus position).
 *   weight_target  device, [V, d_target] bfloat16, row-major, 16-byte
 *                  aligned: the target's output matrix.
 *   hidden_draft   device, [B, K, d_draft] bfloat16 (NULL in greedy mode or
 *                  when K == 0): the draft model's hidden state at the
 *                  position that drew x_i.
 *   weight_draft   device, [V, d_draft] bfloat16 (NULL likewise).
 *   d_target, d_draft  hidden sizes, multiples of 8 (the rows' 16-byte
 *                  alignment), >= 8, < 2^31.
 * Products are exact in float32 and accumulated in float32 over the hidden
 * dimension, so the logits differ from exact ones by float32 accumulation
 * rounding; decisions within the near-tie rule's band may differ from
 * spec_verify run on exactly rounded logits. Other arguments, outputs and
 * errors as spec_verify; the workspace is sv_lmhead_workspace_bytes. A
 * bounded wait inside the GEMM that runs out reports every sequence as
 * SV_SEQ_TIMEOUT. Calls make 3 launches in greedy mode (GEMM, scan, timeout
 * check) and 7 when sampling (GEMM, scan, gather, pair GEMM, two sampler
 * launches, timeout check), plus one memset.
 */
int spec_verify_lmhead(const void* hidden_target, const void* weight_target,
                       const void* hidden_draft, const void* weight_draft,
                       const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                       int64_t d_target, int64_t d_draft, float temperature, uint64_t seed,
                       int mode, int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * spec_verify_lmhead plus the per-row diagnostics of spec_verify_debug (each
 * optional, NULL to skip; sampling mode only, except seq_status).
 */
int spec_verify_lmhead_debug(const void* hidden_target, const void* weight_target,
                             const void* hidden_draft, const void* weight_draft,
                             const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                             int64_t d_target, int64_t d_draft, float temperature, uint64_t seed,
                             int mode, int32_t* out_tokens, int32_t* num_accepted,
                             void* workspace, size_t workspace_bytes, void* stream, double* lse_t,
                             double* lse_d, double* log_ratio, int32_t* seq_status);

/*
 * spec_verify_lmhead with n_events >= 5 cudaEvent_t handles recorded on
 * `stream` before the statistics GEMM, after it, after the scan, after the
 * emitted pairs' GEMM (greedy: after the scan again) and at the end.
 */
int spec_verify_lmhead_timed(const void* hidden_target, const void* weight_target,
                             const void* hidden_draft, const void* weight_draft,
                             const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                             int64_t d_target, int64_t d_draft, float temperature, uint64_t seed,
                             int mode, int32_t* out_tokens, int32_t* num_accepted,
                             void* workspace, size_t workspace_bytes, void* stream,
                             void* const* events, int n_events);

/*
 * Test hook for the timeout paths (no counterpart on the pages):
 * spec_verify_filtered (spec_verify when both cuts are off) with one stage's
 * bulk copies held until the device int32 *gate becomes nonzero:
 *   stage 1  pass 1's producers (with a cut: the thresholds kernel's);
 *   stage 2  the sampler's streaming warps.
 * That wait is bounded like every other wait in the kernels (about 2 s). When
 * it runs out, the held stage marks its work as timed out and returns with no
 * copy in flight, and the sequences it affects are reported as SV_SEQ_TIMEOUT
 * (num_accepted -1, tokens -1, seq_status if given). Stage 1 affects every
 * sequence; stage 2 every sequence the scan found valid. The context stays
 * usable. A caller that sets *gate before the wait runs out gets the ordinary
 * results.
 *   stage  1 or 2 (SV_ERR_ARG otherwise).
 *   gate   device int32, 4-byte aligned (SV_ERR_ARG if NULL, SV_ERR_ALIGN).
 * Other arguments as spec_verify_filtered (workspace: sv_filtered_workspace_bytes,
 * which is sv_workspace_bytes when both cuts are off); seq_status optional.
 */
int spec_verify_gated(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                      float temperature, int64_t top_k, float top_p, uint64_t seed, int mode,
                      int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                      size_t workspace_bytes, void* stream, int32_t* seq_status, int stage,
                      const int32_t* gate);

/*
 * Test hook for the timeout path (no counterpart on the pages): spec_verify_lmhead
 * with the statistics GEMM's producer holding every load until the device
 * int32 *gate becomes nonzero. That wait is bounded like every other wait in
 * the kernels (about 2 s); when it runs out the kernel drains, releases its
 * tensor memory and returns, and every sequence is reported as
 * SV_SEQ_TIMEOUT (num_accepted -1, tokens -1, seq_status if given), with the
 * context still usable. A caller that sets *gate before the wait runs out
 * gets spec_verify_lmhead's results.
 *   gate  device int32, 4-byte aligned (SV_ERR_ARG if NULL, SV_ERR_ALIGN).
 * Other arguments as spec_verify_lmhead_debug (seq_status optional).
 */
int spec_verify_lmhead_gated(const void* hidden_target, const void* weight_target,
                             const void* hidden_draft, const void* weight_draft,
                             const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                             int64_t d_target, int64_t d_draft, float temperature, uint64_t seed,
                             int mode, int32_t* out_tokens, int32_t* num_accepted,
                             void* workspace, size_t workspace_bytes, void* stream,
                             int32_t* seq_status, const int32_t* gate);

/*
 * The LM head alone: out = hidden W^T as float32, the GEMM spec_verify_lmhead
 * runs, exposed so that it can be checked against a plain matrix product.
 *   hidden  device, [R, D] bfloat16, row-major, 16-byte aligned.
 *   weight  device, [V, D] bfloat16, row-major, 16-byte aligned.
 *   D       a multiple of 8, >= 8.
 *   out     device, [R, V] float32, written.
 *   err     device int32, 4-byte aligned: set to 1 (never cleared) when a
 *           bounded wait inside the kernel runs out; out is then incomplete.
 * Stream-ordered; allocates nothing. Returns SV_OK, SV_ERR_ARG, SV_ERR_SIZE
 * (R, V or D >= 2^31), SV_ERR_ALIGN or SV_ERR_CUDA.
 */
int sv_lmhead_logits(const void* hidden, const void* weight, int64_t R, int64_t D, int64_t V,
                     float* out, int32_t* err, void* stream);

/*
 * The Philox4x32-10 generator the verification kernels draw from, evaluated on
 * the device for caller-chosen counters. The pages have no counterpart to this
 * entry point: it exists so that the device generator can be checked word for
 * word against an independent implementation of the published definition
 * (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11: ten rounds of the 4x32 Philox bijection under the key schedule).
 *   seed      the key, (lo32(seed), hi32(seed)), as in spec_verify.
 *   counters  device, [n][4] uint32, 16-byte aligned: counter words x0..x3.
 *   out       device, [n][4] uint32, 16-byte aligned: the four output words
 *             of each counter, written.
 *   n         number of counters, 0 <= n < 2^40; n == 0 enqueues nothing.
 *   stream    cudaStream_t to enqueue on.
 * Stream-ordered; allocates nothing. Returns SV_OK, SV_ERR_ARG (n < 0, or a
 * NULL pointer with n > 0), SV_ERR_SIZE (n too large), SV_ERR_ALIGN or
 * SV_ERR_CUDA.
 */
int sv_philox(uint64_t seed, const uint32_t* counters, uint32_t* out, int64_t n, void* stream);

/* Static description of an SV_* return code. Never NULL. */
const char* sv_error_string(int code);

/* Library ABI version (major * 100 + minor). */
int sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
