// sample.cu -- the token at the emitted position: a draw from the corrected
// distribution after a rejection, or from the bonus row after K acceptances.
//
// What it computes:
//  * "Как работает speculative decoding на уровне логитов..." (aivaro.ru)
//    §5 step 3 / §6 and "Speculative decoding" (aihero.vn), section on
//    accepting by ratio: after a rejection at j the token is drawn from
//    max(0, p_j - q_j) / Z.
//  * Hung-yi Lee, lecture 16 notes, §4 item 4 "The Bonus Token": when all K
//    drafts pass, the token is drawn from the target row K.
// The draw is a two-level exponential race over blocks of kRaceBlock (512)
// tokens. Level 1 picks the block with the largest W_c / E_c, where W_c is the
// sum of the weights w over block c and E_c = -ln v_c, with v_c lane c mod 4 of
// Philox counter (j, b, 1 + c div 4, 1). Level 2 picks the token of that block
// with the largest w_k / E_k, with v_k lane k mod 4 of counter
// (j, b, 1 + k div 4, 0). Uniforms are (2 (word >> 9) + 1) 2^-24, and the
// lowest index wins an exact tie. Block c wins with probability W_c / Z and
// token k within it with w_k / W_c, so the token follows w / Z exactly.
//
// Design: two launches, chained by programmatic dependent launch.
//  * sample_stream_kernel: the emitted row pairs of all sequences are cut into
//    slices of kSliceBytes per row (whole race blocks: two of bf16, one of
//    fp32). A grid of warps, no CTA-wide barriers: each warp takes a
//    contiguous run of slices through its own two-stage ring of bulk copies
//    and writes the weight sum of every race block it covers.
//  * sample_race_kernel: one CTA per sequence runs both levels: level 1 over
//    the block sums (one Philox block per four blocks per thread), then
//    level 2 over the 512 tokens of the winning block, one four-token group
//    per thread, read again from global memory. A kernel of its own keeps this
//    code small and warm in the instruction cache (run inside the streaming
//    kernel, at the end of a warp's run, it stalled on instruction fetches).
//  * Rows that do not start on 16-byte boundaries are copied as the aligned
//    cover of each slice (the last < 16 bytes of a tensor whose size is not a
//    multiple of 16 by element loads) and read one element at a time.
// Weights and block sums are float: a block sum adds at most 512 terms, whose
// rounding stays far inside the 1e-5 near-tie band. The weights carry a factor
// 2^lt common to the row pair (see weight_of). If every residual weight rounded
// to zero, p_j is raced instead.
#include <climits>

#include "sv_device.cuh"
#include "sv_stages.h"

namespace sv {
namespace {

constexpr int kT = kSampleThreads;
constexpr int kWarps = kT / 32;
constexpr int kStageRow = kSliceBytes + 16;   // a slice's bytes plus its 16-byte cover
constexpr int kWarpRing = 2 * 2 * kStageRow;  // two stages of (target | draft)

__device__ __forceinline__ const uint8_t* down16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15));
}
__device__ __forceinline__ const uint8_t* up16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
}

// Slice geometry for one element size.
template <int ES>
struct Geo {
    static constexpr int kEPV = 16 / ES;                // elements per 16-byte vector
    static constexpr int kTok = kSliceBytes / ES;       // tokens per slice
    static constexpr int kBlocks = kTok / kRaceBlock;   // race blocks per slice
    static constexpr int kVPL = kSliceBytes / 16 / 32;  // vectors per lane and row (aligned rows)
    static constexpr int kQPB = kVPL / kBlocks;         // consecutive vectors of a lane per block
    static constexpr int kIPB = kRaceBlock / 32;        // consecutive elements of a lane per block
    static_assert(kTok % kRaceBlock == 0, "a slice holds whole race blocks");
    static_assert(kVPL % kBlocks == 0 && kQPB * 32 * kEPV == kRaceBlock, "vector to block map");
};

// The emitted row pair of one sequence and its normalisers.
struct RowPair {
    const uint8_t* trow;   // target row j
    const uint8_t* drow;   // draft row j, or nullptr for the bonus row
    int32_t j;             // the emitted position (the row index within the sequence)
    float c, mt, md;       // c = log2(e) / T; mt, md: the rows' reference exponents
    float r;               // 2^(lt - ld): the draft term's scale relative to the target's
    float tt, td;          // top-k / top-p thresholds of the two rows (filtered runs)
};

// Sampling weight of one token from its logits, up to a factor common to the
// whole row pair: max(0, p - q) 2^lt after a rejection, p 2^lt for the bonus
// (log2 p = x c - mt - lt, see SeqRecord). Both race levels compare weights of
// one row pair only, so the common factor changes no decision; it saves the
// per-token subtraction of lt and ld. Filtered (F): p and q are the filtered
// rows, 0 below each row's threshold.
template <bool F>
__device__ __forceinline__ float weight_of(const RowPair& rp, float xt, float xd)
{
    float p = ex2(fmaf(xt, rp.c, -rp.mt));
    if (F && !(xt >= rp.tt)) p = 0.f;
    if (rp.drow == nullptr) return p;
    float q = ex2(fmaf(xd, rp.c, -rp.md));
    if (F && !(xd >= rp.td)) q = 0.f;
    return fmaxf(fmaf(-q, rp.r, p), 0.0f);
}

struct Best {
    float score;  // 0 = no candidate yet (every real score is > 0)
    int idx;      // INT_MAX = none
};

__device__ __forceinline__ void take(Best& a, float s, int i)
{
    if (s > a.score || (s == a.score && i < a.idx)) {
        a.score = s;
        a.idx = i;
    }
}

// Best over the warp (largest score, lowest index); every lane gets it.
__device__ __forceinline__ Best warp_best(Best b)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float os = __shfl_xor_sync(0xFFFFFFFFu, b.score, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, b.idx, off);
        take(b, os, oi);
    }
    return b;
}

// Sum over the warp by a fixed butterfly; every lane gets the same value.
__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    return x;
}

__device__ __forceinline__ int64_t lmin(int64_t x, int64_t y) { return x < y ? x : y; }

template <int ES>
__device__ __forceinline__ float elem(const uint8_t* p)
{
    return ES == 2 ? bf16_lo(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)))
                   : *reinterpret_cast<const float*>(p);
}

// One sequence as the sampler sees it.
struct SeqJob {
    RowPair rp;
    int64_t b;
    bool ok;         // the scan found the sequence valid
    bool bad_index;  // its emitted position failed the device-side index check
};

// Reads sequence b's record; returns the emitted position j.
__device__ __forceinline__ int load_seq(SeqJob& s, const SampleArgs& a, int64_t b, int es)
{
    const Geometry& g = a.g;
    const SeqRecord rec = a.seqs[b];
    s.b = b;
    s.ok = rec.status == 0;
    const int64_t K = g.K, row_bytes = g.V * es;
    s.bad_index = s.ok && !SV_IN_RANGE(rec.j, K + 1);
    if (s.bad_index) s.ok = false;
    const RowPairLayout& ly = a.lay;
    s.rp.trow = a.target + (b * ly.t_seq + rec.j * ly.t_pos) * row_bytes;
    s.rp.drow = rec.j < K ? a.draft + (b * ly.d_seq + rec.j * ly.d_pos) * row_bytes : nullptr;
    s.rp.j = rec.j;
    s.rp.c = a.c;
    s.rp.mt = rec.mt;
    s.rp.md = rec.md;
    s.rp.r = rec.j < K ? exp2f(rec.lt - rec.ld) : 1.0f;
    s.rp.tt = rec.tt;
    s.rp.td = rec.td;
    return rec.j;
}

// 16-byte-aligned ends of the target and draft tensors (bulk copies of rows
// that are not 16-byte aligned stop there).
struct TensorEnds {
    const uint8_t* t;
    const uint8_t* d;
};

// The logits of the four tokens k0 .. k0 + 3 (k0 a multiple of 4) of both
// rows, read from global memory (0 past the vocabulary, weighted to 0 below).
template <int ES, bool ALIGNED>
__device__ __forceinline__ void group_load(const SampleArgs& a, const RowPair& rp, int64_t b,
                                           int64_t k0, int64_t V, float (&xt)[4], float (&xd)[4])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) xt[q] = xd[q] = 0.f;
    if (k0 >= V) return;
    if (ALIGNED) {
        // Aligned rows hold a multiple of 16 bytes, so a group that starts
        // inside the row ends inside it (inside one shard: shard widths are
        // multiples of 16 bytes too when the sampler reads shards directly).
        const uint8_t* tb = rp.trow;
        const uint8_t* db = rp.drow;
        int64_t kk = k0;
        if (a.direct) {
            const int64_t Vs = a.g.shard_len;
            const int gi = static_cast<int>(k0 / Vs);
            kk = k0 - gi * Vs;
            tb = a.sh.t[gi] + (b * (a.g.K + 1) + rp.j) * Vs * ES;
            db = rp.drow != nullptr ? a.sh.d[gi] + (b * a.g.K + rp.j) * Vs * ES : nullptr;
        }
        if (ES == 2) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(tb + kk * 2));
            xt[0] = bf16_lo(v.x); xt[1] = bf16_hi(v.x); xt[2] = bf16_lo(v.y); xt[3] = bf16_hi(v.y);
            if (db) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(db + kk * 2));
                xd[0] = bf16_lo(u.x); xd[1] = bf16_hi(u.x); xd[2] = bf16_lo(u.y); xd[3] = bf16_hi(u.y);
            }
        } else {
            const float4 v = __ldg(reinterpret_cast<const float4*>(tb + kk * 4));
            xt[0] = v.x; xt[1] = v.y; xt[2] = v.z; xt[3] = v.w;
            if (db) {
                const float4 u = __ldg(reinterpret_cast<const float4*>(db + kk * 4));
                xd[0] = u.x; xd[1] = u.y; xd[2] = u.z; xd[3] = u.w;
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (k0 + q < V) {
                xt[q] = elem<ES>(rp.trow + (k0 + q) * ES);
                if (rp.drow) xd[q] = elem<ES>(rp.drow + (k0 + q) * ES);
            }
        }
    }
}

// Weights of a loaded group (0 for tokens past the vocabulary).
template <bool F>
__device__ __forceinline__ void group_weights(const RowPair& rp, int64_t k0, int64_t V,
                                              const float (&xt)[4], const float (&xd)[4], float (&w)[4])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = k0 + q < V ? weight_of<F>(rp, xt[q], xd[q]) : 0.f;
}

// Race step over one group of four candidates with weights w (indices
// i0 .. i0 + 3) and clocks from the Philox block of counter ctr.
__device__ __forceinline__ void race_group(Best& best, const float (&w)[4], int64_t i0, uint4 ctr,
                                           uint2 key)
{
    if (!(w[0] > 0.f || w[1] > 0.f || w[2] > 0.f || w[3] > 0.f)) return;
    const uint4 r = philox4x32_10(ctr, key);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (w[q] > 0.f)
            take(best, w[q] / exp_clock(word_to_open_uniform(words[q])), static_cast<int>(i0 + q));
}

// Elements of one 16-byte vector, widened exactly to float.
template <int ES>
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[16 / ES])
{
    if constexpr (ES == 2) {
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    } else {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
}

// Byte offset at which a slice starting at token e0 of `row` lands in its
// stage: 0 for aligned rows, else the row position modulo 16.
template <bool ALIGNED>
__device__ __forceinline__ int stage_offset(const uint8_t* row, int64_t e0, int es)
{
    return ALIGNED ? 0 : static_cast<int>((reinterpret_cast<uintptr_t>(row) + e0 * es) & 15);
}

// Starts the copies of one slice (tokens [e0, e0 + n) of both rows) into a
// stage [target | draft]. Lane 0 issues the bulk copies; for rows that are not
// 16-byte aligned, the bulk copy moves the slice's aligned cover (clipped at
// the tensor's aligned end) and the lanes load the few bytes past that end one
// element at a time. A slice with nothing to read completes the stage's phase
// with a plain arrive.
template <int ES, bool ALIGNED>
__device__ __forceinline__ void issue_slice(const SampleArgs& a, const SeqJob& sj,
                                            const TensorEnds& ends, int64_t e0, int n,
                                            uint8_t* stage, uint64_t* bar, int lane)
{
    if (ALIGNED && a.direct) {
        // Sharded logits: each row's slice [e0, e0 + n) comes from the shards
        // it overlaps, one bulk copy per piece (16-byte aligned: shard widths
        // fill whole vectors and slices start on 2 KB boundaries).
        if (lane == 0) {
            if (!sj.ok || n <= 0) {
                mbar_arrive(bar);
                return;
            }
            const int nrows = sj.rp.drow != nullptr ? 2 : 1;
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nrows * n * ES));
            const int64_t Vs = a.g.shard_len, e1 = e0 + n;
            for (int r = 0; r < nrows; ++r)
                for (int64_t gi = e0 / Vs; gi * Vs < e1; ++gi) {
                    const int64_t p0 = e0 > gi * Vs ? e0 : gi * Vs;
                    const int64_t p1 = e1 < (gi + 1) * Vs ? e1 : (gi + 1) * Vs;
                    const uint8_t* base =
                        r == 0 ? a.sh.t[gi] + (sj.b * (a.g.K + 1) + sj.rp.j) * Vs * ES
                               : a.sh.d[gi] + (sj.b * a.g.K + sj.rp.j) * Vs * ES;
                    bulk_copy_g2s(stage + r * kStageRow + (p0 - e0) * ES, base + (p0 - gi * Vs) * ES,
                                  static_cast<uint32_t>((p1 - p0) * ES), bar);
                }
        }
        return;
    }
    const uint8_t* src[2] = {nullptr, nullptr};
    uint32_t bytes[2] = {0u, 0u};
    if (sj.ok && n > 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint8_t* row = r == 0 ? sj.rp.trow : sj.rp.drow;
            if (row == nullptr) continue;
            const uint8_t* s = row + e0 * ES;
            const uint8_t* e = s + static_cast<int64_t>(n) * ES;
            if (ALIGNED) {
                src[r] = s;
                bytes[r] = static_cast<uint32_t>(n) * ES;
            } else {
                const uint8_t* tend = r == 0 ? ends.t : ends.d;
                const uint8_t* a0 = down16(s);
                const uint8_t* up = up16(e);
                const uint8_t* bend = up < tend ? up : tend;
                const uint32_t bulk = bend > a0 ? static_cast<uint32_t>(bend - a0) : 0u;
                src[r] = a0;
                bytes[r] = bulk;
                uint8_t* dst = stage + r * kStageRow;
                const uint8_t* tail = a0 + bulk > s ? a0 + bulk : s;
                for (const uint8_t* p = tail + lane * ES; p < e; p += 32 * ES) {
                    if (ES == 2)
                        *reinterpret_cast<uint16_t*>(dst + (p - a0)) =
                            __ldg(reinterpret_cast<const unsigned short*>(p));
                    else
                        *reinterpret_cast<uint32_t*>(dst + (p - a0)) =
                            __ldg(reinterpret_cast<const unsigned int*>(p));
                }
            }
        }
    }
    if (lane == 0) {
        const uint32_t tx = bytes[0] + bytes[1];
        if (tx == 0) {
            mbar_arrive(bar);
        } else {
            mbar_arrive_expect_tx(bar, tx);
            if (bytes[0]) bulk_copy_g2s(stage, src[0], bytes[0], bar);
            if (bytes[1]) bulk_copy_g2s(stage + kStageRow, src[1], bytes[1], bar);
        }
    }
}

// Per-lane weight sums of the race blocks of one staged slice of n tokens
// (acc[k]: block k of the slice). Aligned rows: lane l reads vectors
// l, l + 32, ... of each row; other rows: elements l, l + 32, ....
template <int ES, bool ALIGNED, bool F>
__device__ __forceinline__ void sum_slice(const RowPair& rp, const uint8_t* st, int off_t, int off_d,
                                          int n, int lane, float (&acc)[Geo<ES>::kBlocks])
{
    using G = Geo<ES>;
    const uint8_t* bt = st + off_t;
    const uint8_t* bd = st + kStageRow + off_d;
    if (ALIGNED) {
        const int nvec = n / G::kEPV;
#pragma unroll
        for (int q = 0; q < G::kVPL; ++q) {
            const int vi = lane + 32 * q;
            if (vi >= nvec) continue;
            float xt[G::kEPV], xd[G::kEPV];
            unpack<ES>(ld_shared_v4(bt + 16 * vi), xt);
            if (rp.drow)
                unpack<ES>(ld_shared_v4(bd + 16 * vi), xd);
            else
#pragma unroll
                for (int e = 0; e < G::kEPV; ++e) xd[e] = 0.f;
#pragma unroll
            for (int e = 0; e < G::kEPV; ++e) acc[q / G::kQPB] += weight_of<F>(rp, xt[e], xd[e]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < G::kBlocks; ++k) {
#pragma unroll 4
            for (int i = 0; i < G::kIPB; ++i) {
                const int e = lane + 32 * (k * G::kIPB + i);
                if (e >= n) break;
                const float xt = elem<ES>(bt + e * ES);
                const float xd = rp.drow ? elem<ES>(bd + e * ES) : 0.f;
                acc[k] += weight_of<F>(rp, xt, xd);
            }
        }
    }
}

// Lane 0 writes the block sums of one finished slice (NaN: its copy never
// landed).
template <int ES>
__device__ __forceinline__ void store_sums(const SampleArgs& a, int64_t b, int64_t e0, int n,
                                           const float (&sums)[Geo<ES>::kBlocks], int lane)
{
    const int64_t nblk = a.g.nblocks;
    const int64_t c0 = e0 / kRaceBlock;
    const int nb = (n + kRaceBlock - 1) / kRaceBlock;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < Geo<ES>::kBlocks; ++k)
            if (k < nb) a.block_sums[b * nblk + c0 + k] = sums[k];
    }
}

// Launch 1 of 2: a grid of warps over the slices of all sequences' emitted
// row pairs (slice i is slice i mod per_seq of sequence i div per_seq). Each
// warp takes a contiguous run of slices with a two-stage ring: lane 0 copies
// slice i + 1 while the warp sums slice i from the other stage, and writes the
// weight sum of each race block of the slice.
template <int ES, bool ALIGNED, bool F>
__global__ void __launch_bounds__(kT, 3) sample_stream_kernel(const __grid_constant__ SampleArgs a)
{
    using G = Geo<ES>;
    extern __shared__ __align__(128) uint8_t ring[];  // [warp][stage][target | draft]
    __shared__ __align__(8) uint64_t bars[kWarps][2];
    const Geometry& g = a.g;
    const int64_t per_seq = (g.V + G::kTok - 1) / G::kTok;
    const int64_t total = g.B * per_seq;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    // [i0, i1): this warp's slices, split without overflow (w * total can
    // exceed 63 bits at the largest sizes).
    const int64_t qt = total / nwarps, rt = total % nwarps;
    const int64_t i0 = w * qt + (w * rt) / nwarps;
    const int64_t i1 = (w + 1) * qt + ((w + 1) * rt) / nwarps;
    uint8_t* const ring_w = ring + static_cast<size_t>(warp) * kWarpRing;
    auto stage = [&](int st) { return ring_w + st * (2 * kStageRow); };
    if (lane == 0) {
        mbar_init(&bars[warp][0], 1);
        mbar_init(&bars[warp][1], 1);
        fence_barrier_init();
    }
    __syncwarp();
    pdl_wait();  // the scan has finished and the sequence records are visible
    pdl_trigger();  // the race kernel may be scheduled; it waits for this grid
    if (a.gate != nullptr) {
        // Test hook: hold this warp's copies until *gate != 0, bounded like
        // every other wait. Nothing sets it in the tests that use it: the
        // warp then marks its slices with NaN sums (the race kernel reports
        // their sequences as timed out) and returns, with no copy issued.
        int held = 0;
        if (lane == 0) {
            const volatile int32_t* gate = a.gate;
            const long long t0 = clock64();
            while (*gate == 0) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    held = 1;
                    break;
                }
                __nanosleep(1000);
            }
        }
        if (__shfl_sync(0xFFFFFFFFu, held, 0)) {
            const float nan = __uint_as_float(0x7FC00000u);
            float sums[G::kBlocks];
#pragma unroll
            for (int q = 0; q < G::kBlocks; ++q) sums[q] = nan;
            for (int64_t k = i0; k < i1; ++k) {
                const int64_t kb = k / per_seq, ke0 = (k - kb * per_seq) * G::kTok;
                store_sums<ES>(a, kb, ke0, static_cast<int>(lmin(G::kTok, g.V - ke0)), sums, lane);
            }
            return;
        }
    }

    auto tokens_at = [&](int64_t sl) { return static_cast<int>(lmin(G::kTok, g.V - sl * G::kTok)); };
    TensorEnds ends{nullptr, nullptr};
    if (!ALIGNED) {
        ends.t = down16(a.lay.t_end);
        ends.d = a.lay.d_end != nullptr ? down16(a.lay.d_end) : nullptr;
    }
    // Cursor of the next slice to issue: sequence nb, slice nsl of it.
    int64_t nb = i0 / per_seq, nsl = i0 - nb * per_seq;
    SeqJob issued, cur;  // the sequence of the slice issued last / being summed
    issued.b = -1;
    issued.ok = false;
    uint32_t phases = 0;  // bit s: parity of the next phase of stage s
    int64_t i = i0;
    if (i0 < i1) {
        load_seq(issued, a, nb, ES);
        issue_slice<ES, ALIGNED>(a, issued, ends, nsl * G::kTok, tokens_at(nsl), stage(0), &bars[warp][0],
                                 lane);
        __syncwarp();  // element loads into the stage before any lane reads it
    }
    bool failed = false;
    for (; i < i1; ++i) {
        const int s = static_cast<int>((i - i0) & 1);
        cur = issued;
        const int64_t e0 = nsl * G::kTok;
        const int n = tokens_at(nsl);
        if (++nsl == per_seq) {
            nsl = 0;
            ++nb;
        }
        if (i + 1 < i1) {
            if (nb != issued.b) load_seq(issued, a, nb, ES);
            issue_slice<ES, ALIGNED>(a, issued, ends, nsl * G::kTok, tokens_at(nsl), stage(s ^ 1),
                                     &bars[warp][s ^ 1], lane);
        }
        const bool ok = mbar_wait_bounded(&bars[warp][s], (phases >> s) & 1u, nullptr);
        phases ^= 1u << s;
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            break;
        }
        if (cur.ok) {
            float acc[G::kBlocks];
#pragma unroll
            for (int q = 0; q < G::kBlocks; ++q) acc[q] = 0.f;
            sum_slice<ES, ALIGNED, F>(cur.rp, stage(s), stage_offset<ALIGNED>(cur.rp.trow, e0, ES),
                                   cur.rp.drow ? stage_offset<ALIGNED>(cur.rp.drow, e0, ES) : 0, n,
                                   lane, acc);
#pragma unroll
            for (int q = 0; q < G::kBlocks; ++q) acc[q] = warp_sum(acc[q]);
            store_sums<ES>(a, cur.b, e0, n, acc, lane);
        }
        __syncwarp();  // the stage is read out before it is refilled
    }
    if (failed) {
        // A copy did not land in time. Mark this warp's remaining slices with
        // NaN sums, so that the race kernel reports a timeout for their
        // sequences, then let the copies already issued land before the CTA
        // exits.
        const int s = static_cast<int>((i - i0) & 1);
        const float nan = __uint_as_float(0x7FC00000u);
        float sums[G::kBlocks];
#pragma unroll
        for (int q = 0; q < G::kBlocks; ++q) sums[q] = nan;
        for (int64_t k = i; k < i1; ++k) {
            const int64_t kb = k / per_seq, ke0 = (k - kb * per_seq) * G::kTok;
            store_sums<ES>(a, kb, ke0, static_cast<int>(lmin(G::kTok, g.V - ke0)), sums, lane);
        }
        // Stage s: the phase whose wait gave up (its bit was already flipped).
        mbar_wait_bounded(&bars[warp][s], ((phases >> s) & 1u) ^ 1u, nullptr);
        if (i + 1 < i1) mbar_wait_bounded(&bars[warp][s ^ 1], (phases >> (s ^ 1)) & 1u, nullptr);
    }
}

// Level 1 and level 2 of the race run in launch 2, one CTA per sequence: a
// separate small kernel, so that its code stays warm in the instruction cache
// and its CTAs, scheduled while the streaming pass still runs, start the
// moment the block sums are complete.
constexpr int kRaceThreads = kRaceBlock / 4;  // one four-token group per thread
constexpr int kRaceWarps = kRaceThreads / 32;

// Best over the CTA (largest score, lowest index); every thread gets it.
__device__ __forceinline__ Best cta_best(Best b, Best* red)
{
    b = warp_best(b);
    __syncthreads();  // red is free again
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = b;
    __syncthreads();
    Best t = red[0];
#pragma unroll
    for (int i = 1; i < kRaceWarps; ++i) take(t, red[i].score, red[i].idx);
    return t;
}

// Sum over the CTA in a fixed order; every thread gets it.
__device__ __forceinline__ float cta_sum(float x, float* red)
{
    x = warp_sum(x);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float t = red[0];
#pragma unroll
    for (int i = 1; i < kRaceWarps; ++i) t += red[i];
    return t;
}

// Launch 2 of 2: the race of sequence blockIdx.x. Level 1: thread t takes the
// groups of four blocks t, t + kRaceThreads, ... of the block sums (one Philox
// block per group). Level 2: thread t takes four-token group t of the winning
// block. Writes out_tokens[b, j].
template <int ES, bool ALIGNED, bool F>
__global__ void __launch_bounds__(kRaceThreads) sample_race_kernel(const __grid_constant__ SampleArgs a)
{
    __shared__ Best red[kRaceWarps];
    __shared__ float redf[kRaceWarps];
    __shared__ Best s_fb;
    const Geometry& g = a.g;
    const int64_t b = blockIdx.x;
    const int t = threadIdx.x;
    pdl_wait();  // the block sums are complete and visible
    SeqJob sj;
    const int j = load_seq(sj, a, b, ES);
    if (!sj.ok) {
        // The scan wrote the outputs of an invalid sequence; one whose record
        // failed the index check is reported here.
        if (sj.bad_index) {
            for (int64_t i = t; i <= g.K; i += kRaceThreads) a.out_tokens[b * (g.K + 1) + i] = -1;
            if (t == 0) {
                a.num_accepted[b] = -1;
                if (a.seq_status) a.seq_status[b] = kFlagIndex;
            }
        }
        return;
    }
    const int64_t nblk = g.nblocks;
    const float* W = a.block_sums + b * nblk;
    const uint2 key = make_uint2(static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32));
    const uint32_t seq = static_cast<uint32_t>(b), pos = static_cast<uint32_t>(j);

    Best best{0.0f, INT_MAX};
    int nan = 0;
#pragma unroll 1
    for (int64_t gq = t; 4 * gq < nblk; gq += kRaceThreads) {
        float w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t c = 4 * gq + q;
            w[q] = c < nblk ? __ldcg(W + c) : 0.f;
            nan |= !(w[q] == w[q]);  // a wait of the streaming pass gave up
        }
        race_group(best, w, 4 * gq, make_uint4(pos, seq, 1u + static_cast<uint32_t>(gq), 1u), key);
    }
    const bool bad = __syncthreads_or(nan) != 0;
    Best blk = cta_best(best, red);
    if (!bad && blk.idx == INT_MAX) {
        // Every residual weight rounded to zero: race p_j instead (rare; the
        // target row is read once more, block by block).
        sj.rp.drow = nullptr;
        Best fb{0.0f, INT_MAX};
#pragma unroll 1
        for (int64_t c = 0; c < nblk; ++c) {
            const int64_t k0 = c * kRaceBlock + 4 * t;
            float xt[4], xd[4], w[4];
            group_load<ES, ALIGNED>(a, sj.rp, b, k0, g.V, xt, xd);
            group_weights<F>(sj.rp, k0, g.V, xt, xd, w);
            const float sc = cta_sum(((w[0] + w[1]) + w[2]) + w[3], redf);
            if (t == 0 && sc > 0.f) {
                const uint4 r = philox4x32_10(
                    make_uint4(pos, seq, 1u + static_cast<uint32_t>(c >> 2), 1u), key);
                const uint32_t word = (c & 3) == 0 ? r.x : (c & 3) == 1 ? r.y : (c & 3) == 2 ? r.z : r.w;
                take(fb, sc / exp_clock(word_to_open_uniform(word)), static_cast<int>(c));
            }
        }
        if (t == 0) s_fb = fb;
        __syncthreads();
        blk = s_fb;
    }
    Best tok{0.0f, INT_MAX};
    const bool blk_ok = blk.idx == INT_MAX || SV_IN_RANGE(blk.idx, nblk);
    if (!bad && blk_ok && blk.idx != INT_MAX) {
        const int64_t k0 = static_cast<int64_t>(blk.idx) * kRaceBlock + 4 * t;
        float xt[4], xd[4], w[4];
        group_load<ES, ALIGNED>(a, sj.rp, b, k0, g.V, xt, xd);
        group_weights<F>(sj.rp, k0, g.V, xt, xd, w);
        race_group(tok, w, k0, make_uint4(pos, seq, 1u + static_cast<uint32_t>(k0 >> 2), 0u), key);
    }
    tok = cta_best(tok, red);
    const int64_t K1 = g.K + 1;
    const bool idx_ok = blk_ok && (tok.idx == INT_MAX || SV_IN_RANGE(tok.idx, g.V));
    if (bad || !idx_ok || tok.idx == INT_MAX) {
        for (int64_t i = t; i < K1; i += kRaceThreads) a.out_tokens[b * K1 + i] = -1;
        if (t == 0) {
            a.num_accepted[b] = -1;
            if (a.seq_status) a.seq_status[b] = idx_ok ? kFlagTimeout : kFlagIndex;
        }
    } else if (t == 0) {
        a.out_tokens[b * K1 + j] = tok.idx;
    }
}

template <int ES, bool ALIGNED, bool F>
cudaError_t launch_sampler(const SampleArgs& a, cudaStream_t s)
{
    const int smem = kWarps * kWarpRing;
    cudaError_t e = cudaFuncSetAttribute(sample_stream_kernel<ES, ALIGNED, F>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(a.g.pdl != 0, sample_stream_kernel<ES, ALIGNED, F>, dim3(a.g.sample_grid),
                         dim3(kT), static_cast<size_t>(smem), s, a);
    if (e != cudaSuccess) return e;
    return launch_dependent(a.g.pdl != 0, sample_race_kernel<ES, ALIGNED, F>,
                            dim3(static_cast<unsigned>(a.g.B)), dim3(kRaceThreads), 0, s, a);
}

template <bool F>
cudaError_t launch_sampler_f(const SampleArgs& a, cudaStream_t s)
{
    if (a.g.aligned)
        return a.g.es == 2 ? launch_sampler<2, true, F>(a, s) : launch_sampler<4, true, F>(a, s);
    return a.g.es == 2 ? launch_sampler<2, false, F>(a, s) : launch_sampler<4, false, F>(a, s);
}

// Sharded verification: CTA (2 b + r, x) copies a chunk of the emitted target
// (r = 0) or draft (r = 1) row of sequence b from the shards into row 2 b + r
// of the pair buffer. Chunk x covers columns [x C, (x + 1) C) of the logical
// row, C = kGatherThreads vectors; 16-byte copies when every shard row and
// the buffer rows are 16-byte aligned, element copies otherwise.
constexpr int kGatherThreads = 256;

template <int ES>
__global__ void __launch_bounds__(kGatherThreads) gather_pairs_kernel(const __grid_constant__ GatherArgs a)
{
    pdl_wait();  // the scan's sequence records are complete
    const Geometry& g = a.g;
    const int64_t b = blockIdx.x >> 1;
    const int r = blockIdx.x & 1;
    const SeqRecord rec = a.seqs[b];
    if (rec.status != 0 || (r == 1 && rec.j >= g.K)) return;
    const int64_t V = g.V, Vs = g.shard_len, K = g.K;
    uint8_t* dst = a.pairs + (2 * b + r) * V * ES;
    const int64_t row = r == 0 ? b * (K + 1) + rec.j : b * K + rec.j;
    if (g.shard_aligned && g.aligned) {
        constexpr int kEPV = 16 / ES;
        const int64_t nvec = V / kEPV;  // whole vectors: V and Vs are multiples of kEPV
        const int64_t v = static_cast<int64_t>(blockIdx.y) * kGatherThreads + threadIdx.x;
        if (v >= nvec) return;
        const int64_t col = v * kEPV;
        const int gi = static_cast<int>(col / Vs);
        const uint8_t* src = (r == 0 ? a.sh.t[gi] : a.sh.d[gi]) + (row * Vs + (col - gi * Vs)) * ES;
        *reinterpret_cast<uint4*>(dst + col * ES) = __ldg(reinterpret_cast<const uint4*>(src));
    } else {
        const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kGatherThreads * (16 / ES);
        const int64_t c1 = c0 + kGatherThreads * (16 / ES) < V ? c0 + kGatherThreads * (16 / ES) : V;
        for (int64_t col = c0 + threadIdx.x; col < c1; col += kGatherThreads) {
            const int gi = static_cast<int>(col / Vs);
            const uint8_t* src =
                (r == 0 ? a.sh.t[gi] : a.sh.d[gi]) + (row * Vs + (col - gi * Vs)) * ES;
            if (ES == 2)
                *reinterpret_cast<uint16_t*>(dst + col * ES) =
                    __ldg(reinterpret_cast<const unsigned short*>(src));
            else
                *reinterpret_cast<uint32_t*>(dst + col * ES) =
                    __ldg(reinterpret_cast<const unsigned int*>(src));
        }
    }
}

}  // namespace

cudaError_t launch_gather_pairs(const GatherArgs& a, cudaStream_t s)
{
    const int64_t per_chunk = static_cast<int64_t>(kGatherThreads) * (16 / a.g.es);
    const dim3 grid(static_cast<unsigned>(2 * a.g.B),
                    static_cast<unsigned>((a.g.V + per_chunk - 1) / per_chunk));
    return a.g.es == 2 ? launch_dependent(a.g.pdl != 0, gather_pairs_kernel<2>, grid,
                                          dim3(kGatherThreads), 0, s, a)
                       : launch_dependent(a.g.pdl != 0, gather_pairs_kernel<4>, grid,
                                          dim3(kGatherThreads), 0, s, a);
}

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s)
{
    return a.filtered ? launch_sampler_f<true>(a, s) : launch_sampler_f<false>(a, s);
}

int sample_tokens_per_slice(int es) { return es == 2 ? Geo<2>::kTok : Geo<4>::kTok; }

cudaError_t sample_blocks_per_sm(int es, int* blocks)
{
    const int smem = kWarps * kWarpRing;
    auto* k = es == 2 ? sample_stream_kernel<2, false, false> : sample_stream_kernel<4, false, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int b1 = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, k, kT, smem);
    if (e != cudaSuccess) return e;
    auto* ka = es == 2 ? sample_stream_kernel<2, true, false> : sample_stream_kernel<4, true, false>;
    e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int b2 = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, ka, kT, smem);
    if (e != cudaSuccess) return e;
    *blocks = b1 < b2 ? b1 : b2;
    return cudaSuccess;
}

}  // namespace sv
