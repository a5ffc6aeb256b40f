// sv_stages.h -- arguments and launchers of the stages after pass 1 (scan,
// sampler, pair gather, thresholds kernel, LM head). Not part of the public
// ABI; see include/spec_verify.h for that.
#pragma once

#include "sv_internal.h"

namespace sv {

struct FilterArgs {
    const uint8_t* target;
    const uint8_t* draft;
    Geometry g;
    float c;            // log2(e) / T
    int64_t top_k;      // 0 < top_k < V, else off
    float top_p;        // in (0, 1); 1 = off
    FiltRow* rows;      // [B (2K + 1)]
    const int32_t* gate;  // test hook (nullptr in product calls): hold the copies until *gate != 0
};

struct ScanArgs {
    const uint8_t* target;
    const uint8_t* draft;
    const int32_t* tokens;
    Geometry g;
    float c;
    uint64_t seed;
    const Partial* partials;
    int32_t* out_tokens;
    int32_t* num_accepted;
    SeqRecord* seqs;
    double* lse_t;          // optional diagnostics (full pass only)
    double* lse_d;
    double* log_ratio;
    int32_t* seq_status;
    RowMap map;
    // Filtering only (nullptr otherwise): the rows' normalisers and
    // thresholds come from here instead of pass 1's partials.
    const FiltRow* filt;
    float* thr_t;           // optional: thresholds of the target rows [B, K+1]
    float* thr_d;           // and of the draft rows [B, K] (full pass only)
    // Early exit only (nullptr otherwise): the sequences still undecided after
    // this phase, compacted in ascending order by the last CTA to finish.
    int32_t* still;         // [B] per listed sequence: 1 if still undecided
    int32_t* next_active;   // [B]
    int32_t* next_count;    // [1]
    uint32_t* ticket;       // [1], zero before the launch
    Shards sh;
    // LM-head statistics only (0 / nullptr otherwise): the partials are
    // [rows][lm_tiles], one per vocabulary tile, and the draft tokens' raw
    // logits come from tok (row space order) instead of the logits tensors.
    int64_t lm_tiles;
    const float* tok;
};

// Where the sampler finds the emitted row pair: target row j of sequence b is
// row b * t_seq + j * t_pos of `target` (in rows of V elements), the draft row
// likewise. The plain layout is (K + 1, 1) and (K, 1); a gathered pair buffer
// [B][2][V] is (2, 0) with draft = buffer + one row.
struct RowPairLayout {
    int64_t t_seq, t_pos, d_seq, d_pos;
    const uint8_t* t_end;  // end of the target / draft allocation (bulk copies stop
    const uint8_t* d_end;  // at their 16-byte-aligned floor)
};

struct SampleArgs {
    const uint8_t* target;
    const uint8_t* draft;
    Geometry g;
    float c;
    uint64_t seed;
    const SeqRecord* seqs;
    float* block_sums;      // [B][nblocks]: weight of each race block of the emitted row pair
    int32_t* out_tokens;
    int32_t* num_accepted;
    int32_t* seq_status;    // optional
    RowPairLayout lay;
    // Sharded logits with 16-byte-aligned shard widths: the sampler reads
    // the emitted pair from the shards themselves (target row b (K+1) + j of
    // every shard, draft row b K + j), splitting copies at shard boundaries.
    int32_t direct;
    Shards sh;
    int32_t filtered;       // weights are masked by the records' thresholds
    const int32_t* gate;    // test hook (nullptr in product calls): hold the copies until *gate != 0
};

// Sharded verification: copies each sequence's emitted row pair from the
// shards into a contiguous buffer [B][2][V] (the pair the sampler reads).
struct GatherArgs {
    Geometry g;
    Shards sh;
    const SeqRecord* seqs;
    uint8_t* pairs;
};

// LM head on the tensor cores: logits = hidden [R, D] x weights [V, D]^T,
// bfloat16 operands, float32 accumulation, 128 x 256 output tiles. One launch
// covers one or two problems (target and draft heads) over one vocabulary.
//  kLmLogits: float32 logits to out[r * ldo + col].
//  kLmStats:  no logits leave the chip. Sampling: one Partial per (row,
//             vocabulary tile) -- m = ceil(max x c), (hi + lo) 2^m = the tile's
//             sum of 2^(x c) -- and the raw logit of the row's draft token;
//             greedy: the tile's largest logit and its lowest column.
// Rows of problem p are rows row0 + r of the partial / token-logit row space,
// the same space the scan uses: [B (K+1) target rows | B K draft rows].
constexpr int kLmLogits = 0;
constexpr int kLmStats = 1;
struct LmProblem {
    const void* hidden;   // [R, D] bfloat16, 16-byte aligned, D a multiple of 8
    const void* weights;  // [V, D] bfloat16, likewise
    int64_t R;
    int64_t D;
    int64_t row0;         // stats: first row in the row space
    int32_t per;          // stats: rows per sequence (K + 1 target, K draft)
    float* out;           // logits: [R, ldo] float32
    int64_t ldo;
    // Set by launch_lmhead.
    int32_t n_rb, n_kb;
    int64_t tiles;
};
struct LmArgs {
    LmProblem p[2];
    int32_t nprob;
    int64_t V;
    int32_t n_vt;            // set by launch_lmhead
    int32_t K;
    const int32_t* tokens;   // [B, K] (stats, sampling)
    float c;                 // log2(e) / T
    int32_t greedy;
    Partial* part;           // [rows][n_vt] (stats)
    float* tok;              // [rows] token logits (stats, sampling)
    int32_t* err;            // set to 1 when a bounded wait runs out
    // Test hook (nullptr in every product call): the producer holds its
    // loads until *gate != 0, a bounded wait like the others.
    const int32_t* gate;
};

// Launchers (return the launch's cudaError_t).
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);
cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s);
cudaError_t launch_gather_pairs(const GatherArgs& a, cudaStream_t s);
// The thresholds: bfloat16 rows cut by top-p alone or by top-k with k > 64 go
// to the value-count kernel (hist.cu, one CTA on each of `sms` SMs); every
// other cut to the group-maxima kernel (filter.cu, `grid` CTAs).
cudaError_t launch_filter(const FilterArgs& a, int grid, int sms, cudaStream_t s);
cudaError_t launch_hist(const FilterArgs& a, int sms, cudaStream_t s);
// Resident filter CTAs per SM.
cudaError_t filter_blocks_per_sm(int es, int* blocks);
// The LM head; *mapped = false when a tensor map could not be made (nothing
// launched). Vocabulary tiles per row, and the emitted rows' hidden states.
cudaError_t launch_lmhead(int mode, LmArgs a, cudaStream_t s, bool* mapped);
int64_t lmhead_vocab_tiles(int64_t V);
cudaError_t launch_gather_hidden(const void* ht, const void* hd, const SeqRecord* seqs, int64_t B,
                                 int64_t K, int64_t Dt, int64_t Dd, void* out_t, void* out_d,
                                 cudaStream_t s);
cudaError_t launch_lm_fail(const int32_t* err, int64_t B, int64_t K, int32_t* out_tokens,
                           int32_t* num_accepted, int32_t* seq_status, cudaStream_t s);
// Resident sampler CTAs per SM, and the tokens of one sampler slice.
cudaError_t sample_blocks_per_sm(int es, int* blocks);
int sample_tokens_per_slice(int es);

}  // namespace sv
