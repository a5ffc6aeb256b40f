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
// The draw is a two-level exponential race over blocks of kRaceBlock tokens.
// Level 1 picks the block with the largest W_c / E_c, where W_c is the sum of
// the weights w over block c and E_c = -ln v_c, with v_c lane c mod 4 of Philox
// counter (j, b, 1 + c div 4, 1). Level 2 picks the token of that block with the
// largest w_k / E_k, with v_k lane k mod 4 of counter (j, b, 1 + k div 4, 0).
// Uniforms are (2 (word >> 9) + 1) 2^-24, and the lowest index wins an exact
// tie. Block c wins with probability W_c / Z and token k within it with
// w_k / W_c, so the token follows w / Z exactly.
//
// Design. Only the one row pair of each sequence is read again.
//  * Rows on 16-byte boundaries (every vocabulary whose row is a multiple of
//    16 bytes): two launches. sample_stream_kernel is a grid of warps, each
//    taking a contiguous run of 2 KB-per-row slices of the emitted row pairs
//    through its own two-stage ring of bulk copies and writing one float-pair
//    weight sum per slice; it has no atomics and no CTA-wide barriers.
//    sample_finish_kernel, kFinishSplit CTAs per sequence, adds the slice
//    sums of each block in a fixed order and runs level 1 (redundantly, with
//    one result), then each CTA re-reads a quarter of the winning block and
//    races it; the last CTA of the sequence keeps the best quarter.
//  * Other rows: sample_kernel, one CTA per (sequence, block), stages its block
//    in shared memory with bulk copies; the last CTA of a sequence (an atomic
//    ticket: no one waits on it) runs the two levels.
// Weights are float; block sums are float pairs (no float64, which GB300 runs
// at a small fraction of the float32 rate). Per-token random numbers are drawn
// in the winning block only. If every residual weight rounded to zero, p_j is
// raced instead.
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kT = kSampleThreads;
constexpr int kWarps = kT / 32;

// Shared-memory bytes of one staged row block (tokens plus 16-byte cover).
template <int ES>
constexpr int buf_bytes()
{
    return kRaceBlock * ES + 32;
}

__device__ __forceinline__ const uint8_t* down16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15));
}
__device__ __forceinline__ const uint8_t* up16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
}

// Everything about the row pair a CTA works on.
struct RowPair {
    const uint8_t* trow;   // target row j
    const uint8_t* drow;   // draft row j, or nullptr for the bonus row
    const uint8_t* t_end;  // aligned tensor ends
    const uint8_t* d_end;
    float c, mt, lt, md, ld;
    uint64_t seed;
    uint32_t seq, pos;
};

// Sampling weight of one token from its logits: max(0, p - q) after a
// rejection, p for the bonus. log2 p = x c - m - l (see SeqRecord).
__device__ __forceinline__ float weight_of(const RowPair& rp, float xt, float xd)
{
    const float p = ex2(fmaf(xt, rp.c, -rp.mt) - rp.lt);
    if (rp.drow == nullptr) return p;
    const float q = ex2(fmaf(xd, rp.c, -rp.md) - rp.ld);
    return fmaxf(p - q, 0.0f);
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

// One group of four consecutive tokens k0..k0+3 (k0 a multiple of 4) in the
// race of level 2: one Philox block gives their four clocks.
__device__ __forceinline__ void race_group(Best& best, const RowPair& rp, int64_t k0,
                                           const float (&w)[4])
{
    if (!(w[0] > 0.f || w[1] > 0.f || w[2] > 0.f || w[3] > 0.f)) return;
    const uint2 key = make_uint2(static_cast<uint32_t>(rp.seed), static_cast<uint32_t>(rp.seed >> 32));
    const uint4 r = philox4x32_10(
        make_uint4(rp.pos, rp.seq, 1u + static_cast<uint32_t>(k0 >> 2), 0u), key);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (w[q] > 0.f)
            take(best, __fdividef(w[q], exp_clock(word_to_open_uniform(words[q]))),
                 static_cast<int>(k0 + q));
}

// Block-wide float-pair sum over NT threads (fixed tree); every thread gets
// the total.
template <int NT = kT>
__device__ __forceinline__ float2 block_sum2(float hi, float lo, float2* red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
        const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
        float err;
        const float s = two_sum(hi, ohi, &err);
        lo = __fadd_rn(__fadd_rn(lo, olo), err);
        hi = s;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float2(hi, lo);
    __syncthreads();
    float th = red[0].x, tl = red[0].y;
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) {
        float err;
        const float s = two_sum(th, red[i].x, &err);
        tl = __fadd_rn(__fadd_rn(tl, red[i].y), err);
        th = s;
    }
    return make_float2(th, tl);
}

// Block-wide best over NT threads (largest score, lowest index), fixed tree.
template <int NT = kT>
__device__ __forceinline__ Best block_best(Best b, Best* red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float os = __shfl_xor_sync(0xFFFFFFFFu, b.score, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, b.idx, off);
        take(b, os, oi);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = b;
    __syncthreads();
    Best t = red[0];
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) take(t, red[i].score, red[i].idx);
    return t;
}

// ---------------------------------------------------------------------------
// Direct path: rows 16-byte aligned, a span of up to LEN tokens is read with
// 16-byte loads by NT threads; thread t takes vectors t, t + NT, ... (coalesced).
// ---------------------------------------------------------------------------
template <int ES, int NT = kT, int LEN = kRaceBlock>
struct Direct {
    static constexpr int kEPV = 16 / ES;            // elements per vector
    static constexpr int kVPT = LEN / kEPV / NT;    // vectors per thread
    static_assert(LEN % (kEPV * NT) == 0, "span must split evenly over the threads");

    // Elements of one 16-byte vector, widened exactly to float.
    __device__ static __forceinline__ void unpack(const uint4& v, float (&x)[kEPV])
    {
        if constexpr (ES == 2) {
            x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
            x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
        } else {
            x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
            x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
        }
    }

    __device__ static __forceinline__ void load(const RowPair& rp, int64_t e0, int n,
                                                uint4 (&tv)[kVPT], uint4 (&dv)[kVPT])
    {
        const uint4* tp = reinterpret_cast<const uint4*>(rp.trow + e0 * ES);
        const uint4* dp = rp.drow ? reinterpret_cast<const uint4*>(rp.drow + e0 * ES) : nullptr;
        const int nvec = n / kEPV;
#pragma unroll
        for (int q = 0; q < kVPT; ++q) {
            const int vi = static_cast<int>(threadIdx.x) + q * NT;
            tv[q] = vi < nvec ? __ldg(tp + vi) : make_uint4(0, 0, 0, 0);
            dv[q] = (dp != nullptr && vi < nvec) ? __ldg(dp + vi) : make_uint4(0, 0, 0, 0);
        }
    }

    // Per-thread weights of the block (zero past its end).
    __device__ static __forceinline__ void weights(const RowPair& rp, int n, const uint4 (&tv)[kVPT],
                                                   const uint4 (&dv)[kVPT],
                                                   float (&w)[kVPT][kEPV])
    {
        const int nvec = n / kEPV;
#pragma unroll
        for (int q = 0; q < kVPT; ++q) {
            float xt[kEPV], xd[kEPV];
            unpack(tv[q], xt);
            unpack(dv[q], xd);
            const bool in = static_cast<int>(threadIdx.x) + q * NT < nvec;
#pragma unroll
            for (int e = 0; e < kEPV; ++e) w[q][e] = in ? weight_of(rp, xt[e], xd[e]) : 0.f;
        }
    }

    __device__ static float2 block_weight(const RowPair& rp, int64_t e0, int n, float2* red)
    {
        uint4 tv[kVPT], dv[kVPT];
        load(rp, e0, n, tv, dv);
        float w[kVPT][kEPV];
        weights(rp, n, tv, dv, w);
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int q = 0; q < kVPT; ++q)
#pragma unroll
            for (int e = 0; e < kEPV; e += 2) {
                a0 += w[q][e];
                a1 += w[q][e + 1];
            }
        float err;
        const float hi = two_sum(a0, a1, &err);
        return block_sum2<NT>(hi, err, red);
    }

    __device__ static Best race(const RowPair& rp, int64_t e0, int n, Best* red)
    {
        uint4 tv[kVPT], dv[kVPT];
        load(rp, e0, n, tv, dv);
        float w[kVPT][kEPV];
        weights(rp, n, tv, dv, w);
        Best best{0.0f, INT_MAX};
#pragma unroll
        for (int q = 0; q < kVPT; ++q) {
            const int64_t k = e0 + static_cast<int64_t>(threadIdx.x + q * NT) * kEPV;
#pragma unroll
            for (int g = 0; g < kEPV; g += 4) {
                const float wg[4] = {w[q][g], w[q][g + 1], w[q][g + 2], w[q][g + 3]};
                race_group(best, rp, k + g, wg);
            }
        }
        return block_best<NT>(best, red);
    }
};

// ---------------------------------------------------------------------------
// Staged path: rows not 16-byte aligned. The bulk engine moves the aligned
// cover [a0, a0 + bulk) of row bytes [s, e); the last < 16 bytes of a tensor
// whose size is not a multiple of 16 are loaded one element at a time. Byte s
// lands at buf + off.
// ---------------------------------------------------------------------------
struct CopyPlan {
    const uint8_t* a0;
    uint32_t bulk;
    int off;
};

template <int ES>
__device__ __forceinline__ CopyPlan plan_copy(uint8_t* buf, const uint8_t* s, const uint8_t* e,
                                              const uint8_t* tend)
{
    CopyPlan cp;
    cp.a0 = down16(s);
    const uint8_t* up = up16(e);
    const uint8_t* bend = up < tend ? up : tend;
    cp.bulk = bend > cp.a0 ? static_cast<uint32_t>(bend - cp.a0) : 0u;
    cp.off = static_cast<int>(s - cp.a0);
    const uint8_t* tail = bend >= e ? e : (bend > s ? bend : s);
    for (const uint8_t* p = tail + threadIdx.x * ES; p < e; p += kT * ES) {
        if (ES == 2)
            *reinterpret_cast<uint16_t*>(buf + (p - cp.a0)) =
                __ldg(reinterpret_cast<const unsigned short*>(p));
        else
            *reinterpret_cast<uint32_t*>(buf + (p - cp.a0)) =
                __ldg(reinterpret_cast<const unsigned int*>(p));
    }
    return cp;
}

template <int ES>
__device__ __forceinline__ float elem(const uint8_t* p)
{
    return ES == 2 ? bf16_lo(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)))
                   : *reinterpret_cast<const float*>(p);
}

template <int ES>
struct Staged {
    uint8_t* buf_t;
    uint8_t* buf_d;
    uint64_t* bar;
    uint32_t phase;
    int off_t, off_d;

    // Stage block [e0, e0 + n); false if the copy did not land in time.
    __device__ bool stage(const RowPair& rp, int64_t e0, int n)
    {
        const int64_t e1 = e0 + n;
        const CopyPlan ct = plan_copy<ES>(buf_t, rp.trow + e0 * ES, rp.trow + e1 * ES, rp.t_end);
        CopyPlan cd;
        cd.a0 = nullptr;
        cd.bulk = 0;
        cd.off = 0;
        if (rp.drow != nullptr)
            cd = plan_copy<ES>(buf_d, rp.drow + e0 * ES, rp.drow + e1 * ES, rp.d_end);
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(bar, ct.bulk + cd.bulk);
            if (ct.bulk > 0) bulk_copy_g2s(buf_t, ct.a0, ct.bulk, bar);
            if (cd.bulk > 0) bulk_copy_g2s(buf_d, cd.a0, cd.bulk, bar);
        }
        const bool ok = mbar_wait_bounded(bar, phase & 1u, nullptr);
        phase += 1;
        off_t = ct.off;
        off_d = cd.off;
        // Orders the element-wise tail stores before every thread's reads, and
        // agrees on whether the copy landed.
        return __syncthreads_and(ok ? 1 : 0) != 0;
    }

    __device__ float w_at(const RowPair& rp, int e) const
    {
        const float xt = elem<ES>(buf_t + off_t + e * ES);
        const float xd = rp.drow ? elem<ES>(buf_d + off_d + e * ES) : 0.f;
        return weight_of(rp, xt, xd);
    }

    __device__ float2 block_weight(const RowPair& rp, int n, float2* red) const
    {
        float a0 = 0.f;
        for (int e = threadIdx.x; e < n; e += kT) a0 += w_at(rp, e);
        return block_sum2(a0, 0.f, red);
    }

    __device__ Best race(const RowPair& rp, int64_t e0, int n, Best* red) const
    {
        Best best{0.0f, INT_MAX};
        for (int g = threadIdx.x; 4 * g < n; g += kT) {
            float w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = 4 * g + q < n ? w_at(rp, 4 * g + q) : 0.f;
            race_group(best, rp, e0 + 4 * g, w);
        }
        return block_best(best, red);
    }
};

// Level 1: the block with the largest W_c / E_c over blocks with W_c > 0
// (lowest index on a tie); INT_MAX when no block has weight. The flags of all
// block records are OR-ed into *flags.
template <int NT = kT>
__device__ int race_blocks(const volatile ChunkSum* cs, int64_t nch, const RowPair& rp,
                           int* flags, Best* red, int* red_flags)
{
    Best best{0.0f, INT_MAX};
    int fl = 0;
    const uint2 key = make_uint2(static_cast<uint32_t>(rp.seed), static_cast<uint32_t>(rp.seed >> 32));
    for (int64_t c = threadIdx.x; c < nch; c += NT) {
        const float W = cs[c].hi + cs[c].lo;
        fl |= cs[c].flags;
        if (!(W > 0.f)) continue;
        const uint4 r = philox4x32_10(
            make_uint4(rp.pos, rp.seq, 1u + static_cast<uint32_t>(c >> 2), 1u), key);
        const uint32_t lane = static_cast<uint32_t>(c & 3);
        const uint32_t word = lane == 0 ? r.x : lane == 1 ? r.y : lane == 2 ? r.z : r.w;
        take(best, W / exp_clock(word_to_open_uniform(word)), static_cast<int>(c));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red_flags[threadIdx.x >> 5] = fl;
    const Best t = block_best<NT>(best, red);  // its barriers also publish red_flags
    int f = 0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) f |= red_flags[i];
    *flags = f;
    return t.idx;
}

template <int ES, bool STAGED>
__device__ void sample_block(const SampleArgs& a, uint8_t* dyn)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ Best red[kWarps];
    __shared__ float2 red2[kWarps];
    __shared__ int red_flags[kWarps];
    __shared__ int s_last;

    const Geometry& g = a.g;
    const int64_t nch = g.nchunks;
    const int64_t b = blockIdx.x / nch;
    const int64_t c = blockIdx.x - b * nch;
    pdl_wait();  // the scan has finished and the sequence records are visible
    const SeqRecord rec = a.seqs[b];
    if (rec.status != 0) return;

    const int64_t K = g.K, V = g.V;
    const int64_t j = rec.j;
    const int64_t row_bytes = V * ES;
    RowPair rp;
    rp.trow = a.target + (b * (K + 1) + j) * row_bytes;
    rp.t_end = down16(a.target + g.rows_t * row_bytes);
    rp.drow = j < K ? a.draft + (b * K + j) * row_bytes : nullptr;
    rp.d_end = j < K ? down16(a.draft + g.B * K * row_bytes) : nullptr;
    rp.c = a.c;
    rp.mt = rec.mt;
    rp.lt = rec.lt;
    rp.md = rec.md;
    rp.ld = rec.ld;
    rp.seed = a.seed;
    rp.seq = static_cast<uint32_t>(b);
    rp.pos = static_cast<uint32_t>(j);

    Staged<ES> st{dyn, dyn + buf_bytes<ES>(), &bar, 0u, 0, 0};
    if (STAGED) {
        if (threadIdx.x == 0) {
            mbar_init(&bar, 1);
            fence_barrier_init();
        }
        __syncthreads();
    }
    ChunkSum* sums = a.chunk_sums + b * nch;
    auto block_len = [&](int64_t blk) {
        return static_cast<int>(min(static_cast<int64_t>(kRaceBlock), V - blk * kRaceBlock));
    };

    // ---- every CTA: the total weight of its block ----
    float2 W = make_float2(0.f, 0.f);
    int flags = 0;
    const int n = block_len(c);
    if (STAGED) {
        if (st.stage(rp, c * kRaceBlock, n))
            W = st.block_weight(rp, n, red2);
        else
            flags = kFlagTimeout;
    } else {
        W = Direct<ES>::block_weight(rp, c * kRaceBlock, n, red2);
    }
    if (threadIdx.x == 0) {
        ChunkSum cs;
        cs.hi = W.x;
        cs.lo = W.y;
        cs.flags = flags;
        cs.pad = 0;
        sums[c] = cs;
        __threadfence();
        const uint32_t ticket = atomicAdd(&a.tickets[b], 1u);
        s_last = ticket == static_cast<uint32_t>(nch - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- the last CTA of this sequence: level 1 over the blocks ----
    int any_flags = 0;
    bool fallback = false;
    int win = race_blocks(sums, nch, rp, &any_flags, red, red_flags);
    if (any_flags == 0 && win == INT_MAX) {
        // Every residual weight rounded to zero: race p_j instead, block sums first.
        fallback = true;
        rp.drow = nullptr;
        for (int64_t i = 0; i < nch && any_flags == 0; ++i) {
            const int ni = block_len(i);
            float2 Wp = make_float2(0.f, 0.f);
            if (STAGED) {
                if (st.stage(rp, i * kRaceBlock, ni))
                    Wp = st.block_weight(rp, ni, red2);
                else
                    any_flags = kFlagTimeout;
            } else {
                Wp = Direct<ES>::block_weight(rp, i * kRaceBlock, ni, red2);
            }
            if (threadIdx.x == 0) {
                ChunkSum cs;
                cs.hi = Wp.x;
                cs.lo = Wp.y;
                cs.flags = 0;
                cs.pad = 0;
                sums[i] = cs;
            }
            __syncthreads();
        }
        if (any_flags == 0) {
            int f2 = 0;
            win = race_blocks(sums, nch, rp, &f2, red, red_flags);
        }
    }

    // ---- level 2 over the tokens of the winning block ----
    Best tok{0.0f, INT_MAX};
    if (any_flags == 0 && win != INT_MAX) {
        const int64_t p0 = static_cast<int64_t>(win) * kRaceBlock;
        const int np = block_len(win);
        if (STAGED) {
            bool ok = true;
            if (win != c || fallback) ok = st.stage(rp, p0, np);
            if (ok)
                tok = st.race(rp, p0, np, red);
            else
                any_flags = kFlagTimeout;
        } else {
            tok = Direct<ES>::race(rp, p0, np, red);
        }
    }

    if (threadIdx.x == 0) {
        const int64_t K1 = K + 1;
        if (any_flags != 0 || tok.idx == INT_MAX) {
            for (int64_t i = 0; i < K1; ++i) a.out_tokens[b * K1 + i] = -1;
            a.num_accepted[b] = -1;
            if (a.seq_status) a.seq_status[b] = kFlagTimeout;
        } else {
            a.out_tokens[b * K1 + j] = tok.idx;
        }
    }
}

template <int ES, bool STAGED>
__global__ void __launch_bounds__(kT) sample_kernel(const SampleArgs a)
{
    extern __shared__ __align__(128) uint8_t dyn[];
    sample_block<ES, STAGED>(a, dyn);
}

template <int ES, bool STAGED>
cudaError_t launch_one(const SampleArgs& a, cudaStream_t s)
{
    const unsigned grid = static_cast<unsigned>(a.g.B * a.g.nchunks);
    const int smem = STAGED ? 2 * buf_bytes<ES>() : 0;
    if (STAGED) {
        const cudaError_t e = cudaFuncSetAttribute(
            sample_kernel<ES, STAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    return launch_dependent(a.g.pdl != 0, sample_kernel<ES, STAGED>, dim3(grid), dim3(kT), smem, s, a);
}

// ---------------------------------------------------------------------------
// Aligned rows, launch 1 of 2: weight sums of 2 KB-per-row slices.
// ---------------------------------------------------------------------------
template <int ES>
struct Slices {
    static constexpr int kEPV = 16 / ES;                    // elements per vector
    static constexpr int kTok = kSliceBytes / ES;           // tokens per slice
    static constexpr int kPerBlock = kRaceBlock / kTok;     // slices per race block
    static constexpr int kVPL = kSliceBytes / 16 / 32;      // vectors per lane per row
};

__device__ __forceinline__ void warp_sum2(float& hi, float& lo)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
        const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
        float err;
        const float s = two_sum(hi, ohi, &err);
        lo = __fadd_rn(__fadd_rn(lo, olo), err);
        hi = s;
    }
}

__device__ __forceinline__ void row_pair_of(RowPair& rp, const SampleArgs& a, const SeqRecord& rec,
                                            int64_t b, int es)
{
    const Geometry& g = a.g;
    const int64_t K = g.K, row_bytes = g.V * es;
    const int64_t j = rec.j;
    rp.trow = a.target + (b * (K + 1) + j) * row_bytes;
    rp.t_end = down16(a.target + g.rows_t * row_bytes);
    rp.drow = j < K ? a.draft + (b * K + j) * row_bytes : nullptr;
    rp.d_end = j < K ? down16(a.draft + g.B * K * row_bytes) : nullptr;
    rp.c = a.c;
    rp.mt = rec.mt;
    rp.lt = rec.lt;
    rp.md = rec.md;
    rp.ld = rec.ld;
    rp.seed = a.seed;
    rp.seq = static_cast<uint32_t>(b);
    rp.pos = static_cast<uint32_t>(j);
}

// One slice pair as a warp sees it: where its rows are and how many 16-byte
// vectors of each row it holds (0 past the vocabulary).
struct SliceJob {
    RowPair rp;
    bool seq_ok;  // the sequence is valid (else nothing is read or written)
    int nvec;
};

// Slice `sl` of sequence `b`. Consecutive slices of a warp usually share a
// sequence, whose record is then read once.
template <int ES>
__device__ __forceinline__ void slice_job(SliceJob& job, const SampleArgs& a, int64_t b,
                                          int64_t sl, int64_t& cached_b, SliceJob& cache)
{
    using S = Slices<ES>;
    const int64_t e0 = sl * S::kTok;
    if (b != cached_b) {
        cached_b = b;
        const SeqRecord rec = a.seqs[b];
        cache.seq_ok = rec.status == 0;
        if (cache.seq_ok) row_pair_of(cache.rp, a, rec, b, ES);
    }
    job = cache;
    job.nvec = 0;
    if (job.seq_ok && e0 < a.g.V) {
        job.nvec = static_cast<int>(min(static_cast<int64_t>(S::kTok), a.g.V - e0)) / S::kEPV;
        job.rp.trow += e0 * ES;  // point at the slice
        if (job.rp.drow) job.rp.drow += e0 * ES;
    }
}

// Lane 0 starts the bulk copies of a slice pair into a stage; a pair with
// nothing to read completes the stage's phase with a plain arrive.
__device__ __forceinline__ void issue_slice(const SliceJob& job, uint8_t* stage, uint64_t* bar)
{
    const uint32_t bytes = static_cast<uint32_t>(job.nvec) * 16u;
    if (bytes == 0) {
        mbar_arrive(bar);
        return;
    }
    mbar_arrive_expect_tx(bar, job.rp.drow ? 2u * bytes : bytes);
    bulk_copy_g2s(stage, job.rp.trow, bytes, bar);
    if (job.rp.drow) bulk_copy_g2s(stage + kSliceBytes, job.rp.drow, bytes, bar);
}

// Each warp walks a contiguous run of slices with a two-stage ring in shared
// memory: lane 0 copies slice i + 1 (both rows, bulk copies) while the warp
// sums the weights of slice i from the other stage. No registers hold data in
// flight, so every warp keeps a full slice pair moving at all times.
template <int ES>
__global__ void __launch_bounds__(kT) sample_stream_kernel(const SampleArgs a)
{
    using S = Slices<ES>;
    extern __shared__ __align__(128) uint8_t ring[];  // [warp][stage][target | draft]
    __shared__ __align__(8) uint64_t bars[kWarps][2];
    const Geometry& g = a.g;
    const int64_t per_seq = g.nchunks * S::kPerBlock;
    const int64_t total = g.B * per_seq;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    const int64_t i0 = w * total / nwarps, i1 = (w + 1) * total / nwarps;
    uint8_t* stage0 = ring + static_cast<size_t>(warp) * 4 * kSliceBytes;
    uint8_t* stage1 = stage0 + 2 * kSliceBytes;
    if (lane == 0) {
        mbar_init(&bars[warp][0], 1);
        mbar_init(&bars[warp][1], 1);
        fence_barrier_init();
    }
    __syncwarp();
    pdl_wait();  // the scan has finished and the sequence records are visible

    int64_t cached_b = -1;
    SliceJob cache, cur, next;
    cache.seq_ok = false;
    cache.nvec = 0;
    uint32_t phases = 0;  // bit s: parity of the next phase of stage s
    bool failed = false;
    // Cursor (sequence, slice) of the next slice to issue; one division here,
    // increments afterwards.
    int64_t nb = i0 / per_seq, nsl = i0 - nb * per_seq;
    auto advance = [&]() {
        if (++nsl == per_seq) {
            nsl = 0;
            ++nb;
        }
    };
    if (i0 < i1) {
        slice_job<ES>(cur, a, nb, nsl, cached_b, cache);
        if (lane == 0) issue_slice(cur, stage0, &bars[warp][0]);
        advance();
    }
    int64_t i = i0;
    for (; i < i1; ++i) {
        const int s = static_cast<int>((i - i0) & 1);
        uint8_t* buf = s ? stage1 : stage0;
        if (i + 1 < i1) {
            slice_job<ES>(next, a, nb, nsl, cached_b, cache);
            if (lane == 0) issue_slice(next, s ? stage0 : stage1, &bars[warp][s ^ 1]);
            advance();
        }
        const bool ok = mbar_wait_bounded(&bars[warp][s], (phases >> s) & 1u, nullptr);
        phases ^= 1u << s;
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            failed = true;
            break;
        }
        if (cur.seq_ok) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int q = 0; q < S::kVPL; ++q) {
                const int vi = lane + 32 * q;
                if (vi >= cur.nvec) continue;
                float xt[S::kEPV], xd[S::kEPV];
                Direct<ES>::unpack(ld_shared_v4(buf + 16 * vi), xt);
                if (cur.rp.drow)
                    Direct<ES>::unpack(ld_shared_v4(buf + kSliceBytes + 16 * vi), xd);
                else
#pragma unroll
                    for (int e = 0; e < S::kEPV; ++e) xd[e] = 0.f;
#pragma unroll
                for (int e = 0; e < S::kEPV; e += 2) {
                    a0 += weight_of(cur.rp, xt[e], xd[e]);
                    a1 += weight_of(cur.rp, xt[e + 1], xd[e + 1]);
                }
            }
            float lo;
            float hi = two_sum(a0, a1, &lo);
            warp_sum2(hi, lo);
            if (lane == 0) a.slice_sums[i] = make_float2(hi, lo);
        }
        __syncwarp();  // the stage is read out before it is refilled
        cur = next;
    }
    if (failed) {
        // Mark the rest of this warp's slices, then let the copy already
        // issued into the other stage land before the CTA exits.
        const float nan = __uint_as_float(0x7FC00000u);
        for (int64_t k = i + lane; k < i1; k += 32) a.slice_sums[k] = make_float2(nan, nan);
        const int s = static_cast<int>((i - i0) & 1);
        mbar_wait_bounded(&bars[warp][s], ((phases >> s) & 1u) ^ 1u, nullptr);
        if (i + 1 < i1) {
            const int o = s ^ 1;
            mbar_wait_bounded(&bars[warp][o], (phases >> o) & 1u, nullptr);
        }
    }
    pdl_trigger();  // the finish kernel may start launching
}

// ---------------------------------------------------------------------------
// Aligned rows, launch 2 of 2: kFinishSplit CTAs per sequence. Each adds the
// slice sums into block sums and runs level 1 (the same computation, so the
// same winning block, in every CTA of the sequence), then races its quarter
// of the winning block. The last of them to finish (an atomic ticket; no one
// waits) keeps the best of the quarters, the lowest index on a tie.
// ---------------------------------------------------------------------------
template <int ES>
__global__ void __launch_bounds__(kT) sample_finish_kernel(const SampleArgs a)
{
    using S = Slices<ES>;
    constexpr int kQuarter = kRaceBlock / kFinishSplit;
    using DB = Direct<ES, kT, kRaceBlock>;  // whole blocks (zero-residual fall-back)
    using DQ = Direct<ES, kT, kQuarter>;    // one quarter of the winning block
    __shared__ Best red[kWarps];
    __shared__ float2 red2[kWarps];
    __shared__ int red_flags[kWarps];
    __shared__ int s_last;
    const Geometry& g = a.g;
    const int64_t b = blockIdx.x / kFinishSplit;
    const int part = static_cast<int>(blockIdx.x - b * kFinishSplit);
    pdl_wait();  // the slice sums are complete and visible
    const SeqRecord rec = a.seqs[b];
    if (rec.status != 0) return;
    RowPair rp;
    row_pair_of(rp, a, rec, b, ES);
    const int64_t nch = g.nchunks, V = g.V, K1 = g.K + 1;
    ChunkSum* sums = a.chunk_sums + (b * kFinishSplit + part) * nch;  // this CTA's own copy
    auto block_len = [&](int64_t blk) {
        return static_cast<int>(min(static_cast<int64_t>(kRaceBlock), V - blk * kRaceBlock));
    };

    // Block sums: the slice sums of each block, added in slice order.
    for (int64_t c = threadIdx.x; c < nch; c += kT) {
        const float2* sl = a.slice_sums + (b * nch + c) * S::kPerBlock;
        float hi = 0.f, lo = 0.f;
        for (int q = 0; q < S::kPerBlock; ++q) {
            const float2 v = sl[q];
            float err;
            const float s2 = two_sum(hi, v.x, &err);
            lo = __fadd_rn(__fadd_rn(lo, v.y), err);
            hi = s2;
        }
        ChunkSum cs;
        cs.hi = hi;
        cs.lo = lo;
        cs.flags = (hi == hi) ? 0 : kFlagTimeout;  // NaN: a streaming wait gave up
        cs.pad = 0;
        sums[c] = cs;
    }
    __syncthreads();

    int flags = 0;
    int win = race_blocks<kT>(sums, nch, rp, &flags, red, red_flags);
    if (flags != 0) win = INT_MAX;
    if (flags == 0 && win == INT_MAX) {
        // Every residual weight rounded to zero: race p_j instead, block sums first.
        rp.drow = nullptr;
        for (int64_t c = 0; c < nch; ++c) {
            const float2 Wp = DB::block_weight(rp, c * kRaceBlock, block_len(c), red2);
            if (threadIdx.x == 0) {
                ChunkSum cs;
                cs.hi = Wp.x;
                cs.lo = Wp.y;
                cs.flags = 0;
                cs.pad = 0;
                sums[c] = cs;
            }
            __syncthreads();
        }
        win = race_blocks<kT>(sums, nch, rp, &flags, red, red_flags);
    }
    Best tok{0.0f, INT_MAX};
    if (flags == 0 && win != INT_MAX) {
        const int64_t q0 = static_cast<int64_t>(win) * kRaceBlock + part * kQuarter;
        const int nq = static_cast<int>(
            min(static_cast<int64_t>(kQuarter), static_cast<int64_t>(win) * kRaceBlock +
                                                    block_len(win) - q0));
        if (nq > 0) tok = DQ::race(rp, q0, nq, red);
    }

    if (threadIdx.x == 0) {
        FinishPart fp;
        fp.score = tok.score;
        fp.idx = tok.idx;
        fp.flags = flags;
        fp.pad = win == INT_MAX ? 1 : 0;  // level 1 found nothing
        a.parts[b * kFinishSplit + part] = fp;
        __threadfence();
        s_last = atomicAdd(&a.tickets[b], 1u) == static_cast<uint32_t>(kFinishSplit - 1);
    }
    __syncthreads();
    if (!s_last || threadIdx.x != 0) return;
    __threadfence();
    const volatile FinishPart* parts = a.parts + b * kFinishSplit;
    Best best{0.0f, INT_MAX};
    int any_flags = 0, none = 0;
    for (int q = 0; q < kFinishSplit; ++q) {
        take(best, parts[q].score, parts[q].idx);
        any_flags |= parts[q].flags;
        none |= parts[q].pad;
    }
    if (any_flags != 0 || none != 0 || best.idx == INT_MAX) {
        for (int64_t i = 0; i < K1; ++i) a.out_tokens[b * K1 + i] = -1;
        a.num_accepted[b] = -1;
        if (a.seq_status) a.seq_status[b] = kFlagTimeout;
    } else {
        a.out_tokens[b * K1 + rec.j] = best.idx;
    }
}

template <int ES>
cudaError_t launch_direct(const SampleArgs& a, cudaStream_t s)
{
    const int smem = kWarps * 4 * kSliceBytes;
    cudaError_t e = cudaFuncSetAttribute(sample_stream_kernel<ES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(a.g.pdl != 0, sample_stream_kernel<ES>, dim3(a.g.sample_grid), dim3(kT),
                         static_cast<size_t>(smem), s, a);
    if (e != cudaSuccess) return e;
    return launch_dependent(a.g.pdl != 0, sample_finish_kernel<ES>,
                            dim3(static_cast<unsigned>(a.g.B * kFinishSplit)), dim3(kT), 0, s, a);
}

}  // namespace

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s)
{
    if (a.g.aligned) return a.g.es == 2 ? launch_direct<2>(a, s) : launch_direct<4>(a, s);
    return a.g.es == 2 ? launch_one<2, true>(a, s) : launch_one<4, true>(a, s);
}

int sample_slices_per_block(int es) { return es == 2 ? Slices<2>::kPerBlock : Slices<4>::kPerBlock; }

cudaError_t sample_stream_blocks_per_sm(int es, int* blocks)
{
    const int smem = kWarps * 4 * kSliceBytes;
    auto* k = es == 2 ? sample_stream_kernel<2> : sample_stream_kernel<4>;
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k, kT, smem);
}

}  // namespace sv
