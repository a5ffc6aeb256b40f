// filter.cu -- top-k / top-p thresholds of every target and draft row.
//
// What it computes ("Speculative decoding" (aihero.vn), the paragraph on
// temperature, top-k and top-p: whatever transform the draft distribution
// gets, the target distribution gets too): each row's softmax at temperature T
// is cut to the tokens whose logit is >= a threshold and renormalised over
// them. Top-k: the threshold is the k-th largest logit, so every tie at the
// boundary is kept. Top-p, inside the top-k set: the largest logit value v
// whose upper set {x >= v} holds at least top_p of the top-k set's mass. Both
// cuts are thresholds on the logit value: equal logits stay together.
//
// Design: one CTA per row (a persistent grid walks the rows). Thresholds come
// from a radix descent over 32-bit order-preserving keys of the widened
// logits, digits of 12, 12 and 8 bits (bf16 keys are settled after 24 bits:
// their low 16 bits are constant). A level builds, in shared memory, the
// histogram of counts (top-k) and masses (top-p) of the elements that share
// the prefix chosen so far, and picks the digit where the running sum from the
// top reaches its target. Because the top-p threshold is the largest v whose
// upper set reaches top_p times the top-k mass, its descent needs no knowledge
// of the top-k threshold beyond that mass, and shares the top-k histograms
// while both follow the same digits.
//   sweep A (HBM): row maximum, NaN / +inf check, level-1 counts (top-k);
//   sweep B: level-1 masses of the digits at or above the top-k digit, and
//            the level-2 histogram of the top-k digit;
//   further sweeps only where a descent needs a histogram it does not have
//            (level 3 of fp32 rows, or top-p leaving the top-k path).
// Sweeps after A read the row again, normally from L2 (two CTAs per SM keep
// about 300 rows, some 80 MB of bf16 rows of 128K tokens, in flight).
//
// Masses are unsigned 64-bit fixed point: a token's 2^(x c - m), with m the
// ceiling of max x c, scaled by 2^40 and rounded, and accumulated by integer
// atomics, so every sum -- and every decision -- is the same on every run. The
// rounding (at most 2^-41 per token against a row mass >= 1/2) and the SFU
// exponential (a few ulp per term) move a top-p boundary by well under 1e-5 of
// the mass; the sum stays below 2^64 for any V < 2^23.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kFilterThreads = 512;
constexpr int kBins = 4096;   // levels 1 and 2: 12-bit digits
constexpr int kBins3 = 256;   // level 3 (fp32 only): the low 8 bits
constexpr float kFix = 1099511627776.0f;  // 2^40
constexpr size_t kFilterSmem = (2 * kBins + kBins3) * sizeof(uint64_t) +
                               (kBins + kBins3) * sizeof(uint32_t);

// Order-preserving key: x < y  <=>  key(x) < key(y) for non-NaN floats, with
// -0 and +0 one value (they compare equal as logits).
__device__ __forceinline__ uint32_t fkey(float x)
{
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose key is k.
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Fixed-point mass of one token: 2^(x c - m) 2^40, rounded.
__device__ __forceinline__ uint64_t mass_of(float x, float c, float m)
{
    return __float2ull_rn(ex2(fmaf(x, c, -m)) * kFix);
}

template <int ES>
__device__ __forceinline__ float load_elem(const uint8_t* p)
{
    return ES == 2 ? load_logit_bf16(p) : load_logit_f32(p);
}

template <int ES>
__device__ __forceinline__ void unpack_vec(const uint4& v, float (&x)[16 / ES])
{
    if constexpr (ES == 2) {
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    } else {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
}

// Calls f(x) for every element of a row of V logits, spread over the CTA:
// scalar loads up to the first 16-byte boundary and after the last one,
// 16-byte loads in between, four in flight per thread.
template <int ES, typename F>
__device__ __forceinline__ void sweep(const uint8_t* row, int64_t V, F&& f)
{
    constexpr int kEPV = 16 / ES;
    constexpr int kU = 4;
    const uintptr_t p = reinterpret_cast<uintptr_t>(row);
    int64_t head = static_cast<int64_t>(((16u - static_cast<uint32_t>(p & 15u)) & 15u) / ES);
    if (head > V) head = V;
    const int64_t nvec = (V - head) / kEPV;
    const int64_t tail = head + nvec * kEPV;
    const int64_t T = blockDim.x;
    for (int64_t i = threadIdx.x; i < head; i += T) f(load_elem<ES>(row + i * ES));
    const uint4* vp = reinterpret_cast<const uint4*>(row + head * ES);
    int64_t v = threadIdx.x;
    for (; v + (kU - 1) * T < nvec; v += kU * T) {
        uint4 u[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) u[q] = __ldg(vp + v + q * T);
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            float x[kEPV];
            unpack_vec<ES>(u[q], x);
#pragma unroll
            for (int e = 0; e < kEPV; ++e) f(x[e]);
        }
    }
    for (; v < nvec; v += T) {
        float x[kEPV];
        unpack_vec<ES>(__ldg(vp + v), x);
#pragma unroll
        for (int e = 0; e < kEPV; ++e) f(x[e]);
    }
    for (int64_t i = tail + threadIdx.x; i < V; i += T) f(load_elem<ES>(row + i * ES));
}

struct Scratch {
    uint64_t wsum[kFilterThreads / 32];
    float wmax[kFilterThreads / 32];
    uint64_t above;
    int e;
};

template <typename H>
__device__ __forceinline__ void zero(H* h, int n)
{
    for (int i = threadIdx.x; i < n; i += blockDim.x) h[i] = 0;
}

// Largest digit e of h[0, nb) with base + sum_{d >= e} h[d] >= target. Leaves e
// (-1 if even the whole histogram falls short) in s.e and base + sum_{d > e}
// h[d] in s.above. Thread t owns the bins [t per, (t + 1) per); a suffix scan
// over the threads finds the one whose bins hold the crossing. Called by every
// thread of the CTA; integer sums, so the order of the additions is immaterial.
template <typename H>
__device__ void crossing(const H* h, int nb, uint64_t base, uint64_t target, Scratch& s)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int nw = blockDim.x >> 5;
    const int per = nb > static_cast<int>(blockDim.x) ? nb / static_cast<int>(blockDim.x) : 1;
    const int lo = t * per;
    uint64_t local = 0;
    for (int i = 0; i < per; ++i)
        if (lo + i < nb) local += h[lo + i];
    uint64_t incl = local;  // sum over lanes >= lane of this warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t o = __shfl_down_sync(0xFFFFFFFFu, incl, off);
        if (lane + off < 32) incl += o;
    }
    __syncthreads();  // s is free (an earlier call may still read it)
    if (lane == 0) s.wsum[w] = incl;
    if (t == 0) {
        s.e = -1;
        s.above = base;
    }
    __syncthreads();
    uint64_t later = 0;
    for (int v = w + 1; v < nw; ++v) later += s.wsum[v];
    const uint64_t S = base + later + (incl - local);  // everything above this thread's bins
    if (local > 0 && S < target && S + local >= target) {
        uint64_t acc = S;
        for (int i = per - 1; i >= 0; --i) {
            const int d = lo + i;
            if (d >= nb) continue;
            if (acc + h[d] >= target) {
                s.e = d;
                s.above = acc;
                break;
            }
            acc += h[d];
        }
    }
    __syncthreads();
}

// sum_{d >= from} h[d] over the CTA (every thread gets it).
__device__ uint64_t sum_from(const uint64_t* h, int nb, int from, Scratch& s)
{
    uint64_t x = 0;
    for (int d = from + threadIdx.x; d < nb; d += blockDim.x) x += h[d];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s.wsum[threadIdx.x >> 5] = x;
    __syncthreads();
    uint64_t t = 0;
    for (int v = 0; v < static_cast<int>(blockDim.x >> 5); ++v) t += s.wsum[v];
    return t;
}

// Low byte of a bf16 key with the given top digit: keys of positive values
// end in 0x0000, keys of negative values in 0xFFFF.
__device__ __forceinline__ uint32_t bf16_low8(int d1) { return (d1 & 0x800) ? 0x00u : 0xFFu; }

template <int ES>
__global__ void __launch_bounds__(kFilterThreads, 2) filter_kernel(const __grid_constant__ FilterArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t* m1 = reinterpret_cast<uint64_t*>(smem);  // level-1 masses
    uint64_t* m2 = m1 + kBins;                          // level-2 masses
    uint64_t* m3 = m2 + kBins;                          // level-3 masses
    uint32_t* cnt = reinterpret_cast<uint32_t*>(m3 + kBins3);  // level-1, then level-2 counts
    uint32_t* c3 = cnt + kBins;                                // level-3 counts
    __shared__ Scratch s;
    const Geometry& g = a.g;
    const int64_t V = g.V;
    const bool tk = a.top_k > 0 && a.top_k < V;
    const bool tp = a.top_p < 1.0f;
    const uint64_t k = tk ? static_cast<uint64_t>(a.top_k) : 0;
    const float c = a.c;
    pdl_trigger();  // the scan may launch; it waits for this grid before reading

    for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const uint8_t* row =
            r < g.rows_t ? a.target + r * V * ES : a.draft + (r - g.rows_t) * V * ES;
        __syncthreads();  // the previous row is done with the histograms
        if (tk) zero(cnt, kBins);
        __syncthreads();

        // Sweep A: maximum, non-finite values, level-1 counts.
        float mx = __uint_as_float(kF32NegInfBits);
        int bad = 0;
        sweep<ES>(row, V, [&](float x) {
            bad |= (x != x) | (x == __uint_as_float(0x7F800000u));
            mx = fmaxf(mx, x);
            if (tk) atomicAdd(&cnt[fkey(x) >> 20], 1u);
        });
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if ((threadIdx.x & 31) == 0) s.wmax[threadIdx.x >> 5] = mx;
        bad = __syncthreads_or(bad);
        for (int v = 0; v < kFilterThreads / 32; ++v) mx = fmaxf(mx, s.wmax[v]);
        if (bad || mx == __uint_as_float(kF32NegInfBits)) {
            if (threadIdx.x == 0) a.rows[r] = FiltRow{0.f, 0.f, 0.f, kFlagNonFinite};
            continue;
        }
        const float mref = ceilf(mx * c);

        // Top-k, level 1.
        int dk1 = 0;
        uint64_t cab1 = 0;
        if (tk) {
            crossing(cnt, kBins, 0, k, s);
            dk1 = s.e < 0 ? 0 : s.e;
            cab1 = s.above;
            __syncthreads();
            zero(cnt, kBins);
            zero(m2, kBins);
        }
        zero(m1, kBins);
        __syncthreads();

        // Sweep B: level-1 masses at or above the top-k digit, and the top-k
        // digit's level-2 histogram.
        sweep<ES>(row, V, [&](float x) {
            const uint32_t key = fkey(x);
            const int d1 = static_cast<int>(key >> 20);
            if (d1 >= dk1) {
                const uint64_t t = mass_of(x, c, mref);
                if (t) atomicAdd(reinterpret_cast<unsigned long long*>(&m1[d1]), t);
                if (tk && d1 == dk1) {
                    const int d2 = static_cast<int>((key >> 8) & 0xFFFu);
                    atomicAdd(&cnt[d2], 1u);
                    if (t) atomicAdd(reinterpret_cast<unsigned long long*>(&m2[d2]), t);
                }
            }
        });
        __syncthreads();

        uint32_t tau = 0;   // threshold key
        uint64_t mass_k;    // mass of the top-k set
        int dk2 = -1;
        if (tk) {
            crossing(cnt, kBins, cab1, k, s);
            dk2 = s.e < 0 ? 0 : s.e;
            const uint64_t cab2 = s.above;
            const uint64_t above1 = sum_from(m1, kBins, dk1 + 1, s);
            if (ES == 2) {
                tau = (static_cast<uint32_t>(dk1) << 20) | (static_cast<uint32_t>(dk2) << 8) |
                      bf16_low8(dk1);
                mass_k = above1 + sum_from(m2, kBins, dk2, s);
            } else {
                // Level 3: the low 8 bits inside prefix (dk1, dk2).
                zero(c3, kBins3);
                zero(m3, kBins3);
                __syncthreads();
                const uint32_t pre = (static_cast<uint32_t>(dk1) << 12) | static_cast<uint32_t>(dk2);
                sweep<ES>(row, V, [&](float x) {
                    const uint32_t key = fkey(x);
                    if ((key >> 8) == pre) {
                        atomicAdd(&c3[key & 0xFFu], 1u);
                        const uint64_t t = mass_of(x, c, mref);
                        if (t) atomicAdd(reinterpret_cast<unsigned long long*>(&m3[key & 0xFFu]), t);
                    }
                });
                __syncthreads();
                crossing(c3, kBins3, cab2, k, s);
                const int dk3 = s.e < 0 ? 0 : s.e;
                tau = (pre << 8) | static_cast<uint32_t>(dk3);
                mass_k = above1 + sum_from(m2, kBins, dk2 + 1, s) + sum_from(m3, kBins3, dk3, s);
            }
        } else {
            mass_k = sum_from(m1, kBins, 0, s);
        }

        uint64_t kept = mass_k;
        if (tp) {
            const uint64_t tgt =
                static_cast<uint64_t>(ceil(static_cast<double>(a.top_p) * static_cast<double>(mass_k)));
            crossing(m1, kBins, 0, tgt, s);
            const int e1 = s.e < 0 ? dk1 : s.e;
            const uint64_t ab1 = s.above;
            const bool same1 = tk && e1 == dk1;
            if (!same1) {
                __syncthreads();
                zero(m2, kBins);
                __syncthreads();
                sweep<ES>(row, V, [&](float x) {
                    const uint32_t key = fkey(x);
                    if (static_cast<int>(key >> 20) == e1) {
                        const uint64_t t = mass_of(x, c, mref);
                        if (t) atomicAdd(reinterpret_cast<unsigned long long*>(&m2[(key >> 8) & 0xFFFu]), t);
                    }
                });
                __syncthreads();
            }
            crossing(m2, kBins, ab1, tgt, s);
            const int e2 = s.e < 0 ? 0 : s.e;
            const uint64_t ab2 = s.above;
            if (ES == 2) {
                tau = (static_cast<uint32_t>(e1) << 20) | (static_cast<uint32_t>(e2) << 8) |
                      bf16_low8(e1);
                kept = ab2 + m2[e2];
            } else {
                const uint32_t pre = (static_cast<uint32_t>(e1) << 12) | static_cast<uint32_t>(e2);
                if (!(same1 && e2 == dk2)) {
                    __syncthreads();
                    zero(m3, kBins3);
                    __syncthreads();
                    sweep<ES>(row, V, [&](float x) {
                        const uint32_t key = fkey(x);
                        if ((key >> 8) == pre) {
                            const uint64_t t = mass_of(x, c, mref);
                            if (t) atomicAdd(reinterpret_cast<unsigned long long*>(&m3[key & 0xFFu]), t);
                        }
                    });
                    __syncthreads();
                }
                crossing(m3, kBins3, ab2, tgt, s);
                const int e3 = s.e < 0 ? 0 : s.e;
                tau = (pre << 8) | static_cast<uint32_t>(e3);
                kept = s.above + m3[e3];
            }
        }
        if (threadIdx.x == 0) {
            const float thr = tau == 0u ? __uint_as_float(kF32NegInfBits) : key_value(tau);
            const float l = log2f(__ull2float_rn(kept)) - 40.0f;
            a.rows[r] = FiltRow{mref, l, thr, kept > 0 ? 0 : kFlagNonFinite};
        }
    }
}

}  // namespace

cudaError_t launch_filter(const FilterArgs& a, int grid, cudaStream_t s)
{
    auto* k = a.g.es == 2 ? filter_kernel<2> : filter_kernel<4>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kFilterSmem));
    if (e != cudaSuccess) return e;
    return launch_dependent(a.g.pdl != 0, k, dim3(static_cast<unsigned>(grid)), dim3(kFilterThreads),
                            kFilterSmem, s, a);
}

cudaError_t filter_blocks_per_sm(int es, int* blocks)
{
    auto* k = es == 2 ? filter_kernel<2> : filter_kernel<4>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kFilterSmem));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k, kFilterThreads, kFilterSmem);
}

}  // namespace sv
