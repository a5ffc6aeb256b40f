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
// The draw is an exponential race: token = argmax over k with w_k > 0 of
// w_k / E_k, E_k = -ln v_k, v_k the race uniform of token k (lane k mod 4 of
// Philox counter (j, b, 1 + k div 4, 0), mapped to (2 (word >> 9) + 1) 2^-24).
// The first of independent exponential clocks with rates w_k to ring is token
// k with probability w_k / sum(w), so no normaliser and no prefix sum is
// needed; the lowest index wins an exact tie.
//
// Design. Only the one row pair of each sequence is read again. Its V entries
// are cut into chunks of kChunkBytes per row, one CTA per (sequence, chunk).
// A CTA stages its chunk with bulk copies, and each thread races four
// consecutive tokens per Philox call. The block keeps the best (score, index)
// and stores it per chunk. The last CTA of a sequence to finish takes an atomic
// ticket (no one waits on it) and merges the chunk winners in index order. If
// every residual weight rounded to zero, that CTA races p_j over the whole row
// instead.
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kT = kSampleThreads;
constexpr int kWarps = kT / 32;
constexpr int kBufBytes = kChunkBytes + 32;

__device__ __forceinline__ const uint8_t* down16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15));
}
__device__ __forceinline__ const uint8_t* up16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
}

// One row's share of a staged chunk: the bulk engine moves the 16-byte-aligned
// range [a0, a0 + bulk) that covers row bytes [s, e); bytes it cannot take
// (the last < 16 bytes of a tensor whose size is not a multiple of 16) are
// loaded one element at a time. Byte s lands at buf + off.
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

// Everything about the row pair a CTA works on.
struct RowPair {
    const uint8_t* trow;   // target row j
    const uint8_t* drow;   // draft row j, or nullptr for the bonus row
    const uint8_t* t_end;  // aligned tensor ends
    const uint8_t* d_end;
    float c, lt_hi, lt_lo, ld_hi, ld_lo;
    uint64_t seed;
    uint32_t seq, pos;
};

template <int ES>
__device__ __forceinline__ float elem(const uint8_t* p)
{
    return ES == 2 ? bf16_lo(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)))
                   : *reinterpret_cast<const float*>(p);
}

// Weight of staged element e: max(0, p - q) after a rejection, p for the bonus.
template <int ES>
__device__ __forceinline__ float weight(const RowPair& rp, const uint8_t* bt, const uint8_t* bd,
                                        int e)
{
    const float p = ex2(fmaf(elem<ES>(bt + e * ES), rp.c, -rp.lt_hi) - rp.lt_lo);
    if (rp.drow == nullptr) return p;
    const float q = ex2(fmaf(elem<ES>(bd + e * ES), rp.c, -rp.ld_hi) - rp.ld_lo);
    return fmaxf(p - q, 0.0f);
}

// Stage chunk [e0, e1) of the pair; false if the copy did not land in time.
// Thread 0 registers the expected bytes, then issues the copies.
template <int ES>
__device__ bool stage_chunk(const RowPair& rp, int64_t e0, int64_t e1, uint8_t* buf_t,
                            uint8_t* buf_d, uint64_t* bar, uint32_t* phase, int* off_t,
                            int* off_d)
{
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
    const bool ok = mbar_wait_bounded(bar, *phase & 1u, nullptr);
    *phase += 1;
    *off_t = ct.off;
    *off_d = cd.off;
    // Orders the element-wise tail stores before every thread's reads, and
    // agrees on whether the copy landed.
    return __syncthreads_and(ok ? 1 : 0) != 0;
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

// Race the tokens of the staged chunk whose first row index is e0.
template <int ES>
__device__ Best race_chunk(const RowPair& rp, const uint8_t* bt, const uint8_t* bd, int64_t e0,
                           int n)
{
    Best best{0.0f, INT_MAX};
    const uint2 key = make_uint2(static_cast<uint32_t>(rp.seed), static_cast<uint32_t>(rp.seed >> 32));
    for (int g = threadIdx.x; 4 * g < n; g += kT) {
        float w[4];
        bool any = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = 4 * g + q;
            w[q] = e < n ? weight<ES>(rp, bt, bd, e) : 0.0f;
            any |= w[q] > 0.0f;
        }
        if (!any) continue;
        const int64_t k0 = e0 + 4 * g;  // multiple of 4: one Philox block per group
        const uint4 r = philox4x32_10(
            make_uint4(rp.pos, rp.seq, 1u + static_cast<uint32_t>(k0 >> 2), 0u), key);
        const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (!(w[q] > 0.0f)) continue;
            // v in (0, 1), exact in float; E = -ln v, taken as -log1p(v - 1) so
            // that clocks near 0 (v near 1) keep full relative precision.
            const float v = static_cast<float>(2u * (words[q] >> 9) + 1u) * 5.9604644775390625e-8f;
            const float E = -log1pf(v - 1.0f);
            take(best, __fdividef(w[q], E), static_cast<int>(k0 + q));
        }
    }
    return best;
}

// Block-wide best (largest score, lowest index), fixed tree.
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
    for (int i = 1; i < kWarps; ++i) take(t, red[i].score, red[i].idx);
    return t;
}

template <int ES>
__global__ void __launch_bounds__(kT) sample_kernel(const SampleArgs a)
{
    __shared__ __align__(128) uint8_t buf_t[kBufBytes];
    __shared__ __align__(128) uint8_t buf_d[kBufBytes];
    __shared__ __align__(8) uint64_t bar;
    __shared__ Best red[kWarps];
    __shared__ int s_last;

    const Geometry& g = a.g;
    const int64_t nch = g.nchunks;
    const int64_t b = blockIdx.x / nch;
    const int64_t c = blockIdx.x - b * nch;
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
    rp.lt_hi = rec.lse_t_hi;
    rp.lt_lo = rec.lse_t_lo;
    rp.ld_hi = rec.lse_d_hi;
    rp.ld_lo = rec.lse_d_lo;
    rp.seed = a.seed;
    rp.seq = static_cast<uint32_t>(b);
    rp.pos = static_cast<uint32_t>(j);

    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    uint32_t phase = 0;

    const int64_t e0 = c * g.chunk_elems;
    const int64_t e1 = min(e0 + g.chunk_elems, V);
    int off_t = 0, off_d = 0;
    Best mine{0.0f, INT_MAX};
    int flags = 0;
    if (stage_chunk<ES>(rp, e0, e1, buf_t, buf_d, &bar, &phase, &off_t, &off_d))
        mine = race_chunk<ES>(rp, buf_t + off_t, buf_d + off_d, e0, static_cast<int>(e1 - e0));
    else
        flags = kFlagTimeout;
    mine = block_best(mine, red);

    if (threadIdx.x == 0) {
        ChunkBest cb;
        cb.score = mine.score;
        cb.idx = mine.idx;
        cb.flags = flags;
        cb.pad = 0;
        a.chunk_best[b * nch + c] = cb;
        __threadfence();
        const uint32_t ticket = atomicAdd(&a.tickets[b], 1u);
        s_last = ticket == static_cast<uint32_t>(nch - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- the last CTA of this sequence: merge the chunk winners ----
    Best win{0.0f, INT_MAX};
    int any_flags = 0;
    if (threadIdx.x == 0) {
        const volatile ChunkBest* cbs = a.chunk_best + b * nch;
        for (int64_t i = 0; i < nch; ++i) {
            take(win, cbs[i].score, cbs[i].idx);
            any_flags |= cbs[i].flags;
        }
        red[0] = win;
        s_last = any_flags;
    }
    __syncthreads();
    win = red[0];
    any_flags = s_last;
    __syncthreads();

    if (any_flags == 0 && win.idx == INT_MAX) {
        // Every residual weight rounded to zero: race p_j over the whole row.
        rp.drow = nullptr;
        Best all{0.0f, INT_MAX};
        for (int64_t i = 0; i < nch; ++i) {
            const int64_t q0 = i * g.chunk_elems, q1 = min(q0 + g.chunk_elems, V);
            if (!stage_chunk<ES>(rp, q0, q1, buf_t, buf_d, &bar, &phase, &off_t, &off_d)) {
                any_flags = kFlagTimeout;
                break;
            }
            Best cb = race_chunk<ES>(rp, buf_t + off_t, buf_d, q0, static_cast<int>(q1 - q0));
            cb = block_best(cb, red);
            take(all, cb.score, cb.idx);
        }
        win = all;
    }

    if (threadIdx.x == 0) {
        const int64_t K1 = K + 1;
        if (any_flags != 0 || win.idx == INT_MAX) {
            for (int64_t i = 0; i < K1; ++i) a.out_tokens[b * K1 + i] = -1;
            a.num_accepted[b] = -1;
            if (a.seq_status) a.seq_status[b] = kFlagTimeout;
        } else {
            a.out_tokens[b * K1 + j] = win.idx;
        }
    }
}

}  // namespace

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s)
{
    const unsigned grid = static_cast<unsigned>(a.g.B * a.g.nchunks);
    if (a.g.es == 2)
        sample_kernel<2><<<grid, kT, 0, s>>>(a);
    else
        sample_kernel<4><<<grid, kT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sv
