// scan.cu -- the acceptance scan: one CTA per sequence.
//
// What it computes:
//  * "Как работает speculative decoding на уровне логитов..." (aivaro.ru)
//    §5 step 3 and §6, and "Speculative decoding" (aihero.vn), section on
//    accepting by ratio: position i keeps draft token x_i with probability
//    min(1, p_i(x_i) / q_i(x_i)); the first rejection ends the scan and every
//    later draft is dropped. The acceptance draw is u < r with u the lane-0
//    Philox uniform of counter (i, b).
//  * Greedy ("Speculative decoding" (aihero.vn), "Cùng phân bố không có nghĩa
//    cùng chuỗi"): keep x_i while it equals the target row's argmax; the
//    first mismatch emits the argmax itself; all K matching emits the bonus
//    row's argmax (Hung-yi Lee, lecture 16 notes, §4 item 4).
//
// It merges pass 1's per-warp partials of the sequence's rows, a warp per
// row, in a fixed order (float pairs, exact power-of-two rescales), so the
// result does not depend on timing. The log-domain acceptance test is float32:
// GB300 runs float64 at a small fraction of the float32 rate, and the float32
// error, about 1e-6 on the ratio, is far inside the 1e-5 near-tie band. Only
// the optional diagnostic outputs are widened to double. Everything the
// sampler needs (the emitted position j and the normalisers of row j) goes to
// the SeqRecord.
#include <climits>

#include "sv_device.cuh"
#include "sv_stages.h"

namespace sv {
namespace {

constexpr int kScanMaxThreads = 544;  // a warp per row, up to 17 rows per round
constexpr double kLn2 = 0.69314718055994530942;

// CTAs pass 1 used: at most one per tile (every range non-empty).
__device__ __forceinline__ int64_t used_grid(int64_t tiles, const Geometry& g)
{
    return tiles < g.grid ? tiles : g.grid;
}

// The pass-1 CTA whose tile range [c T / G, (c + 1) T / G) holds tile t.
__device__ __forceinline__ int cta_of_tile(int64_t t, int64_t tiles, const Geometry& g)
{
    return static_cast<int>(((t + 1) * used_grid(tiles, g) - 1) / tiles);
}

// Merge the partials of one row, one warp per row: lane l takes partials
// l, l + 32, ... (online), then the lanes combine over a fixed butterfly.
// Sampling -> the row's log2 normaliser as (m, l): integer-valued exponent m
// and l = log2 of the float-pair sum; greedy -> argmax. Every lane returns the
// same values. thr: the row's top-k / top-p threshold (-inf: unfiltered).
struct RowNorm {
    float m;
    float l;
    float thr;
};

__device__ void merge_row(const ScanArgs& a, int64_t lrow, int64_t tiles, int lane, RowNorm* norm,
                          int* argmax, int* flags)
{
    const Geometry& g = a.g;
    int fl = 0;
    float M = __uint_as_float(kF32NegInfBits), hi = 0.f, lo = 0.f;
    float best = __uint_as_float(kF32NegInfBits);
    int idx = INT_MAX;
    auto take = [&](const Partial& p) {
        fl |= p.flags;
        if (g.mode == 0) {
            merge_scaled(M, hi, lo, p.m, p.hi, p.lo);
        } else {
            const int pi = __float_as_int(p.hi);
            if (p.m > best || (p.m == best && pi < idx)) {
                best = p.m;
                idx = pi;
            }
        }
    };
    // LM-head statistics: one partial per vocabulary tile, in tile order.
    for (int64_t q = lane; q < a.lm_tiles; q += 32) take(a.partials[lrow * a.lm_tiles + q]);
    // Pass 1: the logical row's shard rows, in shard order (one pass-1 row
    // when not sharded); each one's partials in CTA, then warp order.
    for (int64_t row = lrow * g.row_shards; a.lm_tiles == 0 && row < (lrow + 1) * g.row_shards;
         ++row) {
        const int64_t t0 = row * g.tiles_per_row;
        const int c0 = cta_of_tile(t0, tiles, g);
        const int c1 = cta_of_tile(t0 + g.tiles_per_row - 1, tiles, g);
        const int n = (c1 - c0 + 1) * kRowConsumerWarps;
        for (int q = lane; q < n; q += 32) {
            const int c = c0 + q / kRowConsumerWarps;
            const int w = q % kRowConsumerWarps;
            const int64_t first =
                (static_cast<int64_t>(c) * tiles / used_grid(tiles, g)) / g.tiles_per_row;
            take(a.partials[(static_cast<int64_t>(c) * g.maxseg + (row - first)) * kRowConsumerWarps +
                            w]);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, off);
        if (g.mode == 0) {
            const float om = __shfl_xor_sync(0xFFFFFFFFu, M, off);
            const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
            const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
            merge_scaled(M, hi, lo, om, ohi, olo);
        } else {
            const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, off);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, idx, off);
            if (ob > best || (ob == best && oi < idx)) {
                best = ob;
                idx = oi;
            }
        }
    }
    if (g.mode == 0) {
        // log2(hi + lo) = log2(hi) + lo / (hi ln 2) to first order (|lo| <= 2^-24 hi).
        const float l = log2f(hi) + lo / (hi * 0.69314718055994531f);
        const bool ok = M > __uint_as_float(kF32NegInfBits) && M < __uint_as_float(0x7F800000u) &&
                        hi > 0.f && l < __uint_as_float(0x7F800000u);
        // All -inf, or a sum that is not finite; a row that timed out in
        // pass 1 reports only the timeout.
        if (!ok && !(fl & kFlagTimeout)) fl |= kFlagNonFinite;
        norm->m = M;
        norm->l = l;
        norm->thr = __uint_as_float(kF32NegInfBits);
    } else {
        *argmax = (idx == INT_MAX) ? 0 : idx;  // a row of -inf only: index 0
    }
    *flags = fl;
}

template <int ES>
__device__ __forceinline__ float load_logit(const uint8_t* p)
{
    return ES == 2 ? load_logit_bf16(p) : load_logit_f32(p);
}

// Compaction for early exit, run by the last CTA of the launch: the listed
// sequences whose `still` flag is set, in list order (a block-wide prefix sum
// in fixed order, so the next list is the same on every run).
__device__ void compact_still(const ScanArgs& a, int64_t nseq)
{
    __shared__ int warp_tot[32];
    __shared__ int s_carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < nseq; base += blockDim.x) {
        const int64_t sq = base + threadIdx.x;
        const int f = sq < nseq ? __ldcg(a.still + sq) : 0;
        int incl = f;  // inclusive scan within the warp
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int before = s_carry;
        for (int w = 0; w < warp; ++w) before += warp_tot[w];
        if (f) {
            const int32_t id = a.map.active != nullptr ? a.map.active[sq] : static_cast<int32_t>(sq);
            a.next_active[before + incl - 1] = id;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int t = 0;
            for (int w = 0; w < nwarps; ++w) t += warp_tot[w];
            s_carry += t;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) *a.next_count = s_carry;
}

// One CTA per listed sequence (the full pass lists every sequence). The phase
// covers positions [p0, p0 + npos) that carry a draft token, npos =
// min(nt, K - p0), and the bonus row K when p0 + nt = K + 1. The CTA merges
// the phase's rows, takes the phase's decisions, and then either decides the
// sequence (first rejection at j in the phase, or the bonus after K
// acceptances) or leaves it undecided for the next phase.
template <int ES>
__global__ void __launch_bounds__(kScanMaxThreads, 2) scan_kernel(const __grid_constant__ ScanArgs a)
{
    // Dynamic shared memory: [nt + nd] row normalisers (sampling) or argmaxes
    // (greedy, in .m), then the phase's draft tokens and their target / draft
    // logits.
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_status;
    __shared__ int s_j;
    __shared__ int s_last;
    const Geometry& g = a.g;
    const RowMap& m = a.map;
    const bool phased = m.count != nullptr;
    int64_t nseq = g.B;
    if (phased) {
        pdl_wait();  // the previous scan's list, and this phase's pass 1, are complete
        nseq = *m.count;
    }
    const int64_t sq = blockIdx.x;
    if (sq >= nseq) return;
    const int64_t b = m.active != nullptr ? m.active[sq] : sq;
    if (!SV_IN_RANGE(b, a.g.B)) return;  // a listed sequence outside the batch: nothing to report to
    const int64_t K = g.K, V = g.V;
    const bool sampling = g.mode == 0;
    const int p0 = m.p0;
    const int npos = static_cast<int>(min(static_cast<int64_t>(m.nt), K - p0));
    const bool has_bonus = p0 + m.nt == K + 1;
    const int nrows = m.nt + m.nd;
    RowNorm* sh = reinterpret_cast<RowNorm*>(smem_raw);
    int32_t* sx = reinterpret_cast<int32_t*>(sh + nrows);
    float* stx = reinterpret_cast<float*>(sx + npos);
    float* sdx = stx + npos;
    if (threadIdx.x == 0) {
        s_status = 0;
        s_j = p0 + npos;  // no rejection among the phase's positions
    }
    __syncthreads();

    // Inputs only (complete before pass 1 started): the draft tokens and the
    // logits they select. In the full pass this overlaps the tail of pass 1.
    // Every token is checked once, in the phase that starts at position 0.
    if (p0 == 0)
        for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
            const int32_t x = a.tokens[b * K + i];
            if (x < 0 || static_cast<int64_t>(x) >= V) atomicOr(&s_status, kFlagBadToken);
        }
    for (int q = threadIdx.x; q < npos; q += blockDim.x) {
        const int64_t i = p0 + q;
        const int32_t x = a.tokens[b * K + i];
        sx[q] = x;
        if (x >= 0 && static_cast<int64_t>(x) < V && sampling && a.tok != nullptr) {
            stx[q] = a.tok[b * (K + 1) + i];
            sdx[q] = a.tok[g.B * (K + 1) + b * K + i];
        } else if (x >= 0 && static_cast<int64_t>(x) < V && sampling) {
            // Token x lives in shard x / Vs, at column x mod Vs.
            const int64_t Vs = g.shard_len;
            const int gi = static_cast<int>(x / Vs);
            const int64_t col = x - gi * Vs;
            stx[q] = load_logit<ES>(a.sh.t[gi] + ((b * (K + 1) + i) * Vs + col) * ES);
            sdx[q] = load_logit<ES>(a.sh.d[gi] + ((b * K + i) * Vs + col) * ES);
        }
    }
    pdl_trigger();  // the next kernel may start launching
    if (!phased) pdl_wait();  // pass 1 has finished and its partials are visible
    __syncthreads();

    const int64_t tiles = map_rows(m, nseq) * g.row_shards * g.tiles_per_row;
    const int lane = threadIdx.x & 31;
    for (int q = threadIdx.x >> 5; q < nrows; q += blockDim.x >> 5) {
        const int64_t row = q < m.nt ? sq * m.nt + q : nseq * m.nt + sq * m.nd + (q - m.nt);
        RowNorm nm{0.f, 0.f, 0.f};
        int am = 0, fl = 0;
        if (!SV_IN_RANGE(row, nseq * nrows)) {
            fl = kFlagIndex;
        } else if (a.filt != nullptr) {
            const FiltRow fr = a.filt[row];
            nm = RowNorm{fr.m, fr.l, fr.thr};
            fl = fr.flags;
        } else {
            merge_row(a, row, tiles, lane, &nm, &am, &fl);
        }
        if (lane == 0) {
            if (!sampling) nm.m = __int_as_float(am);
            sh[q] = nm;
            if (fl) atomicOr(&s_status, fl);
        }
    }
    __syncthreads();

    if (s_status == 0) {
        for (int q = threadIdx.x; q < npos; q += blockDim.x) {
            const int32_t x = sx[q];
            const int64_t i = p0 + q;
            bool reject;
            if (sampling) {
                const RowNorm nt = sh[q], nd = sh[m.nt + q];
                // log2 p_i(x) and log2 q_i(x): the fma is exact before its one
                // rounding, and the normaliser's parts enter separately. A
                // token below a row's threshold has probability 0 there; one
                // the (filtered) target gives 0 is rejected.
                const bool in_t = stx[q] >= nt.thr, in_d = sdx[q] >= nd.thr;
                const float ninf = __uint_as_float(kF32NegInfBits);
                const float lp2 = in_t ? fmaf(stx[q], a.c, -nt.m) - nt.l : ninf;
                const float lq2 = in_d ? fmaf(sdx[q], a.c, -nd.m) - nd.l : ninf;
                const float lr2 = lp2 - lq2;
                if (a.log_ratio) a.log_ratio[b * K + i] = static_cast<double>(lr2) * kLn2;
                const float r = !in_t ? 0.f : (lr2 >= 0.f ? 1.f : ex2(lr2));
                const float u = word_to_uniform(
                    verify_random_words(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i)).x);
                reject = !(u < r);
            } else {
                reject = __float_as_int(sh[q].m) != x;
            }
            if (reject) atomicMin(&s_j, static_cast<int>(i));
        }
    }
    __syncthreads();

    const int status = s_status;
    const int j = s_j;
    const bool decided = status != 0 || j < p0 + npos || has_bonus;
    if (sampling && !phased) {
        for (int q = threadIdx.x; q < m.nt; q += blockDim.x)
            if (a.thr_t) a.thr_t[b * (K + 1) + q] = sh[q].thr;
        for (int q = threadIdx.x; q < m.nd; q += blockDim.x)
            if (a.thr_d) a.thr_d[b * K + q] = sh[m.nt + q].thr;
        for (int q = threadIdx.x; q < m.nt; q += blockDim.x)
            if (a.lse_t)
                a.lse_t[b * (K + 1) + q] =
                    (static_cast<double>(sh[q].m) + static_cast<double>(sh[q].l)) * kLn2;
        for (int q = threadIdx.x; q < m.nd; q += blockDim.x)
            if (a.lse_d)
                a.lse_d[b * K + q] = (static_cast<double>(sh[m.nt + q].m) +
                                      static_cast<double>(sh[m.nt + q].l)) *
                                     kLn2;
    }
    int32_t* out = a.out_tokens + b * (K + 1);
    if (status != 0) {
        for (int64_t i = threadIdx.x; i <= K; i += blockDim.x) out[i] = -1;
    } else {
        // Positions of this phase up to j keep their drafts; after a
        // decision every later position is padding.
        for (int64_t i = p0 + threadIdx.x; i <= K; i += blockDim.x) {
            if (i < j && i < p0 + npos)
                out[i] = sx[i - p0];
            else if (decided && i > j)
                out[i] = -1;
            else if (decided && i == j && !sampling)
                out[i] = __float_as_int(sh[j - p0].m);
        }
    }
    if (threadIdx.x == 0) {
        if (decided) {
            a.num_accepted[b] = status != 0 ? -1 : j;
            if (a.seq_status) a.seq_status[b] = status;
            if (sampling) {
                SeqRecord rec;
                rec.j = j;
                rec.status = status;
                rec.mt = rec.lt = rec.md = rec.ld = 0.f;
                rec.tt = rec.td = __uint_as_float(kF32NegInfBits);
                if (status == 0) {
                    rec.mt = sh[j - p0].m;
                    rec.lt = sh[j - p0].l;
                    rec.tt = sh[j - p0].thr;
                    if (j < K) {
                        rec.md = sh[m.nt + j - p0].m;
                        rec.ld = sh[m.nt + j - p0].l;
                        rec.td = sh[m.nt + j - p0].thr;
                    }
                }
                a.seqs[b] = rec;
            }
        }
        if (a.next_active != nullptr) {
            a.still[sq] = decided ? 0 : 1;
            __threadfence();  // the flag before the ticket
            s_last = atomicAdd(a.ticket, 1u) == static_cast<uint32_t>(nseq - 1);
        }
    }
    if (a.next_active == nullptr) return;
    __syncthreads();
    if (!s_last) return;
    __threadfence();  // every other CTA's flag after the ticket
    compact_still(a, nseq);
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s)
{
    const int64_t nrows = a.map.nt + a.map.nd;
    const int64_t npos = a.map.nt < a.g.K - a.map.p0 ? a.map.nt : a.g.K - a.map.p0;
    const size_t smem = sizeof(RowNorm) * static_cast<size_t>(nrows) + 12 * static_cast<size_t>(npos);
    // A warp per row, at most 17 (the headline's 2K + 1 rows; more take a
    // second round): the launch bounds keep two such CTAs on an SM.
    const int warps = static_cast<int>(nrows < 2 ? 2 : (nrows > 17 ? 17 : nrows));
    const dim3 grid(static_cast<unsigned>(a.g.B)), block(32 * warps);
    return a.g.es == 2 ? launch_dependent(a.g.pdl != 0, scan_kernel<2>, grid, block, smem, s, a)
                       : launch_dependent(a.g.pdl != 0, scan_kernel<4>, grid, block, smem, s, a);
}

}  // namespace sv
