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
// It merges pass 1's per-warp partials of the sequence's rows in a fixed
// order (double precision, exact power-of-two rescales), so the result does
// not depend on timing. The log-domain acceptance test is done in double.
// Everything the sampler needs (the emitted position j and the two
// normalisers of row j as float pairs) goes to the SeqRecord, and the
// sampler's ticket counter for the sequence is reset here.
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kScanThreads = 128;
constexpr double kLn2 = 0.69314718055994530942;

__device__ __forceinline__ int cta_of_tile(int64_t t, const Geometry& g)
{
    return static_cast<int>(((t + 1) * g.grid - 1) / g.tiles);
}

// Merge the partials of one row: sampling -> (log2 normaliser, flags);
// greedy -> (argmax, flags).
__device__ void merge_row(const ScanArgs& a, int64_t row, double* lse2, int* argmax, int* flags)
{
    const Geometry& g = a.g;
    const int64_t t0 = row * g.tiles_per_row;
    const int c0 = cta_of_tile(t0, g);
    const int c1 = cta_of_tile(t0 + g.tiles_per_row - 1, g);
    int fl = 0;
    if (g.mode == 0) {
        float M = __uint_as_float(kF32NegInfBits);
        for (int c = c0; c <= c1; ++c) {
            const int64_t first = (static_cast<int64_t>(c) * g.tiles / g.grid) / g.tiles_per_row;
            const Partial* p = a.partials +
                               (static_cast<int64_t>(c) * g.maxseg + (row - first)) * kRowConsumerWarps;
            for (int w = 0; w < kRowConsumerWarps; ++w) {
                M = fmaxf(M, p[w].m);
                fl |= p[w].flags;
            }
        }
        double S = 0.0;
        if (M != __uint_as_float(kF32NegInfBits)) {
            for (int c = c0; c <= c1; ++c) {
                const int64_t first =
                    (static_cast<int64_t>(c) * g.tiles / g.grid) / g.tiles_per_row;
                const Partial* p = a.partials + (static_cast<int64_t>(c) * g.maxseg + (row - first)) *
                                                    kRowConsumerWarps;
                for (int w = 0; w < kRowConsumerWarps; ++w) S += p[w].s * pow2_neg_int_d(p[w].m - M);
            }
        }
        const double l = static_cast<double>(M) + log2(S);
        if (!(l > -1e300 && l < 1e300)) fl |= kFlagNonFinite;  // all -inf, +inf or NaN
        *lse2 = l;
    } else {
        float best = __uint_as_float(kF32NegInfBits);
        int idx = INT_MAX;
        for (int c = c0; c <= c1; ++c) {
            const int64_t first = (static_cast<int64_t>(c) * g.tiles / g.grid) / g.tiles_per_row;
            const Partial* p = a.partials +
                               (static_cast<int64_t>(c) * g.maxseg + (row - first)) * kRowConsumerWarps;
            for (int w = 0; w < kRowConsumerWarps; ++w) {
                const int pi = static_cast<int>(p[w].s);
                fl |= p[w].flags;
                if (p[w].m > best || (p[w].m == best && pi < idx)) {
                    best = p[w].m;
                    idx = pi;
                }
            }
        }
        *argmax = (idx == INT_MAX) ? 0 : idx;  // a row of -inf only: index 0
    }
    *flags = fl;
}

template <int ES>
__device__ __forceinline__ float load_logit(const uint8_t* p)
{
    return ES == 2 ? load_logit_bf16(p) : load_logit_f32(p);
}

__device__ __forceinline__ void split_hi_lo(double x, float* hi, float* lo)
{
    *hi = static_cast<float>(x);
    *lo = static_cast<float>(x - static_cast<double>(*hi));
}

template <int ES>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanArgs a)
{
    extern __shared__ double sh[];  // [2K+1]: log2 normalisers, or argmaxes (greedy)
    __shared__ int s_status;
    __shared__ int s_j;
    const Geometry& g = a.g;
    const int64_t b = blockIdx.x;
    const int64_t K = g.K, V = g.V;
    const bool sampling = g.mode == 0;
    const int64_t nrows = sampling ? 2 * K + 1 : K + 1;
    if (threadIdx.x == 0) {
        s_status = 0;
        s_j = static_cast<int>(K);
    }
    __syncthreads();

    for (int64_t q = threadIdx.x; q < nrows; q += blockDim.x) {
        const int64_t row = q <= K ? b * (K + 1) + q : g.rows_t + b * K + (q - K - 1);
        double l = 0.0;
        int am = 0, fl = 0;
        merge_row(a, row, &l, &am, &fl);
        sh[q] = sampling ? l : static_cast<double>(am);
        if (fl) atomicOr(&s_status, fl);
    }
    for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
        const int32_t x = a.tokens[b * K + i];
        if (x < 0 || static_cast<int64_t>(x) >= V) atomicOr(&s_status, kFlagBadToken);
    }
    __syncthreads();

    const double cd = static_cast<double>(a.c);
    if (s_status == 0) {
        for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
            const int32_t x = a.tokens[b * K + i];
            bool reject;
            if (sampling) {
                const float tx = load_logit<ES>(a.target + ((b * (K + 1) + i) * V + x) * ES);
                const float dx = load_logit<ES>(a.draft + ((b * K + i) * V + x) * ES);
                const double lp2 = static_cast<double>(tx) * cd - sh[i];
                const double lq2 = static_cast<double>(dx) * cd - sh[K + 1 + i];
                const double lr2 = lp2 - lq2;
                if (a.log_ratio) a.log_ratio[b * K + i] = lr2 * kLn2;
                const double r = lr2 >= 0.0 ? 1.0 : exp2(lr2);
                const double u = word_to_uniform(
                    verify_random_words(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(i)).x);
                reject = !(u < r);
            } else {
                reject = static_cast<int64_t>(sh[i]) != static_cast<int64_t>(x);
            }
            if (reject) atomicMin(&s_j, static_cast<int>(i));
        }
    }
    __syncthreads();

    const int status = s_status;
    const int j = s_j;
    if (sampling) {
        for (int64_t q = threadIdx.x; q <= K; q += blockDim.x)
            if (a.lse_t) a.lse_t[b * (K + 1) + q] = sh[q] * kLn2;
        for (int64_t q = threadIdx.x; q < K; q += blockDim.x)
            if (a.lse_d) a.lse_d[b * K + q] = sh[K + 1 + q] * kLn2;
    }
    int32_t* out = a.out_tokens + b * (K + 1);
    if (status != 0) {
        for (int64_t i = threadIdx.x; i <= K; i += blockDim.x) out[i] = -1;
    } else {
        for (int64_t i = threadIdx.x; i <= K; i += blockDim.x) {
            if (i < j)
                out[i] = a.tokens[b * K + i];
            else if (i > j)
                out[i] = -1;
            else if (!sampling)
                out[i] = static_cast<int32_t>(sh[i]);
        }
    }
    if (threadIdx.x == 0) {
        a.num_accepted[b] = status != 0 ? -1 : j;
        if (a.seq_status) a.seq_status[b] = status;
        if (sampling) {
            SeqRecord rec;
            rec.j = j;
            rec.status = status;
            rec.lse_t_hi = rec.lse_t_lo = rec.lse_d_hi = rec.lse_d_lo = 0.f;
            rec.pad[0] = rec.pad[1] = 0;
            if (status == 0) {
                split_hi_lo(sh[j], &rec.lse_t_hi, &rec.lse_t_lo);
                if (j < K) split_hi_lo(sh[K + 1 + j], &rec.lse_d_hi, &rec.lse_d_lo);
            }
            a.seqs[b] = rec;
            a.tickets[b] = 0u;
        }
    }
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s)
{
    const size_t smem = sizeof(double) * static_cast<size_t>(2 * a.g.K + 1);
    if (a.g.es == 2)
        scan_kernel<2><<<static_cast<unsigned>(a.g.B), kScanThreads, smem, s>>>(a);
    else
        scan_kernel<4><<<static_cast<unsigned>(a.g.B), kScanThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sv
