// sv_internal.h -- layouts shared by the library's translation units and
// pass 1's arguments (not part of the public ABI; see include/spec_verify.h
// for that). The later stages' arguments and launchers are in sv_stages.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace sv {

// ---------------------------------------------------------------------------
// Row statistics (pass 1). Each CTA streams a contiguous range of fixed-size
// tiles of the concatenated row space [target rows | draft rows] through a
// STAGES-deep ring of shared-memory buffers filled by bulk copies. One warp
// issues the copies; kRowConsumerWarps warps reduce.
// ---------------------------------------------------------------------------
constexpr int kRowTileBytes = 32768;
constexpr int kRowStages = 3;
constexpr int kRowConsumerWarps = 16;
constexpr int kRowThreads = (kRowConsumerWarps + 1) * 32;

// Residual / bonus sampling (pass 3): a two-level exponential race over
// blocks of kRaceBlock tokens of the emitted row pair. The block length is part
// of the sampler's definition (it decides which random numbers are drawn), not
// a tuning knob. The sampler streams the row pairs in slices of kSliceBytes per
// row, one warp per slice (a slice holds whole race blocks), then races each
// sequence in a CTA of its own.
constexpr int kRaceBlock = 512;
constexpr int kSampleThreads = 256;
constexpr int kSliceBytes = 2048;

constexpr int kMaxK = 1024;

// Flags carried by partial results and sequence records.
constexpr int kFlagNonFinite = 2;  // == SV_SEQ_NONFINITE
constexpr int kFlagTimeout = 4;    // == SV_SEQ_TIMEOUT
constexpr int kFlagBadToken = 1;   // == SV_SEQ_BAD_TOKEN
constexpr int kFlagIndex = 8;      // == SV_SEQ_INDEX (device-side index checks)

// One warp's reduction of one row segment.
//   sampling: (hi + lo) * 2^m = sum over the segment of 2^(x*c), kept as a float
//             pair scaled by an integer-valued reference exponent m (log2
//             units), m = -inf and hi = lo = 0 when the segment is all -inf.
//   greedy:   m = largest raw logit, hi = its lowest index (int bits), or
//             2^31 - 1 when no element beat -inf.
//   flags:    kFlagNonFinite / kFlagTimeout.
// No double precision: GB300 runs float64 at a small fraction of its float32
// rate, so sums that need more than 24 bits are carried as float pairs.
struct Partial {
    float m;
    float hi;
    float lo;
    int32_t flags;
};
static_assert(sizeof(Partial) == 16, "Partial layout");

// Per-sequence record written by the acceptance scan, read by the sampler.
// A row's log2 normaliser log2 sum_k 2^(x_k c) is m + l: m the integer-valued
// reference exponent, l = log2 of the scaled sum.
//
// With top-k / top-p filtering the normalisers are those of the kept tokens,
// and tt / td are the rows' thresholds: token k keeps its probability when
// its logit is >= the threshold, else gets 0 (-inf: no filtering).
struct SeqRecord {
    int32_t j;         // emitted position (0..K)
    int32_t status;    // SV_SEQ_* bits; 0 = valid
    float mt, lt;      // normaliser of target row j
    float md, ld;      // normaliser of draft row j (unused when j == K)
    float tt, td;      // thresholds of target / draft row j
};
static_assert(sizeof(SeqRecord) == 32, "SeqRecord layout");

struct Geometry {
    int64_t B, K, V;
    int32_t es;             // bytes per element (4 or 2)
    int32_t mode;           // SV_SAMPLE / SV_GREEDY
    int64_t rows_t;         // target rows = B (K + 1)
    int64_t rows;           // rows streamed in pass 1 (target, then draft when sampling)
    int64_t tile_elems;     // elements per pass-1 tile
    int64_t tiles_per_row;
    int64_t tiles;          // rows * tiles_per_row
    int32_t grid;           // pass-1 CTAs
    int32_t maxseg;         // most row segments one pass-1 CTA can touch
    int32_t aligned;        // every full row (V elements) starts on a 16-byte boundary
    int64_t shard_len;      // Vs, the shard width (V when not sharded)
    int32_t shards;         // G (1 when not sharded)
    int32_t shard_aligned;  // Vs elements fill whole 16-byte vectors
    int32_t row_shards;     // pass-1 rows per logical row: 1, or G when shard rows are
                            // not 16-byte aligned or shorter than 4 KB (then pass 1
                            // streams each shard row)
    int64_t row_len;        // pass-1 row length: V, or Vs when row_shards == G
    int32_t row_aligned;    // pass-1 rows fill whole 16-byte vectors
    int64_t nblocks;        // race blocks per row
    int32_t sample_grid;    // CTAs of the sampler
    int32_t pdl;            // chain the kernels with programmatic dependent launch
};

// The rows one pass-1 launch and its scan cover. The full pass: every row of
// every sequence (active == nullptr, count == nullptr, p0 = 0, nt = K + 1,
// nd = K or 0 in greedy mode). Early exit: the rows of positions
// [p0, p0 + nt) (target) and [p0, p0 + nd) (draft) of the sequences still
// undecided, listed in ascending order by the previous scan. The row space is
// [n * nt target rows | n * nd draft rows], sequence-major within each part.
struct RowMap {
    const int32_t* active;  // sequence ids of the phase; nullptr = 0 .. B - 1
    const int32_t* count;   // how many (device memory); nullptr = B
    int32_t p0;             // first position of the phase
    int32_t nt;             // target rows per sequence in the phase
    int32_t nd;             // draft rows per sequence in the phase
};

__host__ __device__ __forceinline__ int64_t map_rows(const RowMap& m, int64_t n)
{
    return n * (m.nt + m.nd);
}

// The vocabulary split into G shards of Vs columns (a tensor-parallel LM
// head's output): shard g of every row holds tokens [g Vs, (g + 1) Vs).
// Without sharding G = 1 and shard 0 is the whole tensor. When Vs fills whole
// 16-byte vectors, pass 1 tiles the logical rows and splits a tile's bulk copy
// at the shard boundaries; otherwise it streams each logical row as G shard
// rows (consecutive in its row space) and the scan merges them.
constexpr int kMaxShards = 16;
struct Shards {
    const uint8_t* t[kMaxShards];  // target shards [B, K+1, Vs]
    const uint8_t* d[kMaxShards];  // draft shards [B, K, Vs] (unused in greedy mode)
};

// Top-k / top-p filtering: one record per row of the row space [target rows
// b (K+1) + i | draft rows B (K+1) + b K + i]. The filtered row keeps the
// tokens whose logit is >= thr and renormalises over them: log2 p'(x) =
// x c - m - l for those, with m an integer-valued reference exponent and l
// = log2 of the kept mass scaled by 2^-m.
struct FiltRow {
    float m;
    float l;
    float thr;
    int32_t flags;  // kFlagNonFinite: NaN or +inf in the row, or no finite logit
};
static_assert(sizeof(FiltRow) == 16, "FiltRow layout");

struct RowStatsArgs {
    const uint8_t* target;
    const uint8_t* draft;
    Geometry g;
    float c;                // log2(e) / T
    Partial* partials;      // [grid][maxseg][kRowConsumerWarps]
    RowMap map;
    Shards sh;
    // Test hook (nullptr in every product call): the producer holds its
    // copies until *gate != 0, a bounded wait like the others.
    const int32_t* gate;
};

// Launch with programmatic stream serialization (the kernel must call
// pdl_wait() before it reads what the previous kernel in the stream wrote).
// With pdl == false it is an ordinary launch (the wait then returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                             size_t smem, cudaStream_t s, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Pass 1 (the other stages' arguments and launchers are in sv_stages.h).
cudaError_t launch_row_stats(const RowStatsArgs& a, cudaStream_t s);
// Resident pass-1 CTAs per SM for this dtype / mode (occupancy query).
cudaError_t row_stats_blocks_per_sm(int es, int mode, int* blocks);

}  // namespace sv
