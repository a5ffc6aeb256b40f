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
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kScanMaxThreads = 1024;  // a warp per row, up to 32 rows per round
constexpr double kLn2 = 0.69314718055994530942;

__device__ __forceinline__ int cta_of_tile(int64_t t, const Geometry& g)
{
    return static_cast<int>(((t + 1) * g.grid - 1) / g.tiles);
}

// Merge the partials of one row, one warp per row: lane l takes partials
// l, l + 32, ... (online), then the lanes combine over a fixed butterfly.
// Sampling -> the row's log2 normaliser as (m, l): integer-valued exponent m
// and l = log2 of the float-pair sum; greedy -> argmax. Every lane returns the
// same values.
struct RowNorm {
    float m;
    float l;
};

__device__ void merge_row(const ScanArgs& a, int64_t row, int lane, RowNorm* norm, int* argmax,
                          int* flags)
{
    const Geometry& g = a.g;
    const int64_t t0 = row * g.tiles_per_row;
    const int c0 = cta_of_tile(t0, g);
    const int c1 = cta_of_tile(t0 + g.tiles_per_row - 1, g);
    const int n = (c1 - c0 + 1) * kRowConsumerWarps;
    int fl = 0;
    float M = __uint_as_float(kF32NegInfBits), hi = 0.f, lo = 0.f;
    float best = __uint_as_float(kF32NegInfBits);
    int idx = INT_MAX;
    for (int q = lane; q < n; q += 32) {
        const int c = c0 + q / kRowConsumerWarps;
        const int w = q % kRowConsumerWarps;
        const int64_t first = (static_cast<int64_t>(c) * g.tiles / g.grid) / g.tiles_per_row;
        const Partial p =
            a.partials[(static_cast<int64_t>(c) * g.maxseg + (row - first)) * kRowConsumerWarps + w];
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
        if (!ok) fl |= kFlagNonFinite;  // all -inf, or a sum that is not finite
        norm->m = M;
        norm->l = l;
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

template <int ES>
__global__ void __launch_bounds__(kScanMaxThreads, 1) scan_kernel(const ScanArgs a)
{
    // Dynamic shared memory: [2K+1] row normalisers (sampling) or argmaxes
    // (greedy, in .m), then the K draft tokens and their target / draft logits.
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ int s_status;
    __shared__ int s_j;
    const Geometry& g = a.g;
    const int64_t b = blockIdx.x;
    const int64_t K = g.K, V = g.V;
    const bool sampling = g.mode == 0;
    const int64_t nrows = sampling ? 2 * K + 1 : K + 1;
    RowNorm* sh = reinterpret_cast<RowNorm*>(smem_raw);
    int32_t* sx = reinterpret_cast<int32_t*>(sh + (2 * K + 1));
    float* stx = reinterpret_cast<float*>(sx + K);
    float* sdx = stx + K;
    if (threadIdx.x == 0) {
        s_status = 0;
        s_j = static_cast<int>(K);
    }
    __syncthreads();

    // Inputs only (complete before pass 1 started): the draft tokens and the
    // logits they select. This overlaps the tail of pass 1.
    for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
        const int32_t x = a.tokens[b * K + i];
        sx[i] = x;
        if (x < 0 || static_cast<int64_t>(x) >= V) {
            atomicOr(&s_status, kFlagBadToken);
        } else if (sampling) {
            stx[i] = load_logit<ES>(a.target + ((b * (K + 1) + i) * V + x) * ES);
            sdx[i] = load_logit<ES>(a.draft + ((b * K + i) * V + x) * ES);
        }
    }
    pdl_trigger();  // the sampler's first kernel may start launching
    pdl_wait();     // pass 1 has finished and its partials are visible
    __syncthreads();

    const int lane = threadIdx.x & 31;
    for (int64_t q = threadIdx.x >> 5; q < nrows; q += blockDim.x >> 5) {
        const int64_t row = q <= K ? b * (K + 1) + q : g.rows_t + b * K + (q - K - 1);
        RowNorm nm{0.f, 0.f};
        int am = 0, fl = 0;
        merge_row(a, row, lane, &nm, &am, &fl);
        if (lane == 0) {
            if (!sampling) nm.m = __int_as_float(am);
            sh[q] = nm;
            if (fl) atomicOr(&s_status, fl);
        }
    }
    __syncthreads();

    if (s_status == 0) {
        for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
            const int32_t x = sx[i];
            bool reject;
            if (sampling) {
                const RowNorm nt = sh[i], nd = sh[K + 1 + i];
                // log2 p_i(x) and log2 q_i(x): the fma is exact before its one
                // rounding, and the normaliser's parts enter separately.
                const float lp2 = fmaf(stx[i], a.c, -nt.m) - nt.l;
                const float lq2 = fmaf(sdx[i], a.c, -nd.m) - nd.l;
                const float lr2 = lp2 - lq2;
                if (a.log_ratio) a.log_ratio[b * K + i] = static_cast<double>(lr2) * kLn2;
                const float r = lr2 >= 0.f ? 1.f : ex2(lr2);
                const float u = word_to_uniform(
                    verify_random_words(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i)).x);
                reject = !(u < r);
            } else {
                reject = __float_as_int(sh[i].m) != x;
            }
            if (reject) atomicMin(&s_j, static_cast<int>(i));
        }
    }
    __syncthreads();

    const int status = s_status;
    const int j = s_j;
    if (sampling) {
        for (int64_t q = threadIdx.x; q <= K; q += blockDim.x)
            if (a.lse_t)
                a.lse_t[b * (K + 1) + q] =
                    (static_cast<double>(sh[q].m) + static_cast<double>(sh[q].l)) * kLn2;
        for (int64_t q = threadIdx.x; q < K; q += blockDim.x)
            if (a.lse_d)
                a.lse_d[b * K + q] = (static_cast<double>(sh[K + 1 + q].m) +
                                      static_cast<double>(sh[K + 1 + q].l)) *
                                     kLn2;
    }
    int32_t* out = a.out_tokens + b * (K + 1);
    if (status != 0) {
        for (int64_t i = threadIdx.x; i <= K; i += blockDim.x) out[i] = -1;
    } else {
        for (int64_t i = threadIdx.x; i <= K; i += blockDim.x) {
            if (i < j)
                out[i] = sx[i];
            else if (i > j)
                out[i] = -1;
            else if (!sampling)
                out[i] = __float_as_int(sh[i].m);
        }
    }
    if (threadIdx.x == 0) {
        a.num_accepted[b] = status != 0 ? -1 : j;
        if (a.seq_status) a.seq_status[b] = status;
        if (sampling) {
            SeqRecord rec;
            rec.j = j;
            rec.status = status;
            rec.mt = rec.lt = rec.md = rec.ld = 0.f;
            rec.pad[0] = rec.pad[1] = 0;
            if (status == 0) {
                rec.mt = sh[j].m;
                rec.lt = sh[j].l;
                if (j < K) {
                    rec.md = sh[K + 1 + j].m;
                    rec.ld = sh[K + 1 + j].l;
                }
            }
            a.seqs[b] = rec;
        }
    }
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s)
{
    const size_t smem = sizeof(RowNorm) * static_cast<size_t>(2 * a.g.K + 1) + 12 * static_cast<size_t>(a.g.K);
    const int64_t rows = a.g.mode == 0 ? 2 * a.g.K + 1 : a.g.K + 1;
    const int warps = static_cast<int>(rows < 2 ? 2 : (rows > 32 ? 32 : rows));
    const dim3 grid(static_cast<unsigned>(a.g.B)), block(32 * warps);
    return a.g.es == 2 ? launch_dependent(a.g.pdl != 0, scan_kernel<2>, grid, block, smem, s, a)
                       : launch_dependent(a.g.pdl != 0, scan_kernel<4>, grid, block, smem, s, a);
}

}  // namespace sv
