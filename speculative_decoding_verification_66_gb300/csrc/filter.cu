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
// Design: one CTA per row (a persistent grid walks the rows). The exact
// thresholds come from a radix select over 32-bit order-preserving keys of
// the widened logits, 8 bits per level, with shared-memory histograms of
// counts (top-k) and masses (top-p), one copy per warp so that lanes of
// different warps never contend. Run over a whole row, that select would cost
// some twenty instructions and a contended atomic per element -- several
// times the HBM budget -- so it runs on a short list of candidates instead:
//  * first read (HBM): each thread keeps the maximum of each lane position
//    of its 16-byte vectors (NaN-propagating packed max: half an instruction
//    per bf16 element), which gives the row maximum, the NaN / +inf check and
//    4096 (bf16) or 2048 (fp32) group maxima of disjoint groups.
//  * top-k (k up to the number of groups, with or without top-p): the k-th
//    largest group maximum, to 16 bits, bounds the k-th largest logit from
//    below. A second read (from L2) compares packed pairs against the bound
//    and appends the few elements at or above it -- about k -- to the list,
//    which then holds the whole top-k set.
//  * top-p alone: the second read adds each element's mass into per-thread
//    private bins (no atomics) by its log2 distance from the row maximum,
//    32 bins of one unit; the bin where the running mass from the top reaches
//    top_p times the row mass is read again into the list, or, when it holds
//    too many elements, split into 32 sub-bins the same way, up to three times.
//  * anything else (larger k, a list that overflows, a crossing in the
//    bins' far tail) runs the radix select over the whole row.
// Sweeps after the first read the row again, normally from L2 (two CTAs per SM
// keep about 300 rows, some 80 MB of bf16 rows of 128K tokens, in flight).
//
// Masses are integers, so every sum -- and every decision -- is the same on
// every run: a list element's mass is its 2^(x c - m) (m the ceiling of
// max x c) scaled by 2^40 and rounded; a bin adds per-thread 32-bit sums of
// its elements' masses relative to the bin's upper edge, scaled by 2^SC with
// SC chosen so that a thread's sum cannot overflow, and rescaled by a shift.
// The roundings (below 2^-22 of each element's mass) and the SFU exponential
// (a few ulp per term) move a top-p boundary by well under 1e-5 of the mass.
#include <cooperative_groups.h>

#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

namespace cg = cooperative_groups;

constexpr int kFilterThreads = 512;
constexpr int kWarpsF = kFilterThreads / 32;
constexpr int kListCap = 6144;                       // list entries (keys)
constexpr int kDBins = 32;                           // log2-distance bins per level
constexpr int kRefine = 3;                           // sub-bin levels after the first
constexpr int kRadixBins = 256;                      // 8-bit digits
constexpr float kFix = 1099511627776.0f;             // 2^40

// Group maxima per thread: one per lane position of a 16-byte vector.
template <int ES>
constexpr int groups() { return 16 / ES; }

// Dynamic shared memory: the per-thread bins [kDBins][kFilterThreads]; on the
// top-k path and in every select, the same 64 KB hold the candidate keys
// (first 16 KB), the per-warp counts (next 16 KB) and the per-warp masses
// (last 32 KB). Then the list.
constexpr size_t kBinsBytes = sizeof(uint32_t) * kDBins * kFilterThreads;
constexpr size_t kCandBytes = 16384;
constexpr size_t kCountBytes = sizeof(uint32_t) * kWarpsF * kRadixBins;
constexpr size_t kMassBytes = sizeof(uint64_t) * kWarpsF * kRadixBins;
constexpr size_t kListBytes = sizeof(uint32_t) * kListCap;
constexpr size_t kFilterSmem = kBinsBytes + kListBytes;
static_assert(kCandBytes + kCountBytes + kMassBytes <= kBinsBytes, "select scratch fits the bins");
static_assert(sizeof(uint32_t) * kFilterThreads * 8 <= kCandBytes, "candidates fit");

// Order-preserving key: x < y  <=>  key(x) < key(y) for non-NaN floats, with
// -0 and +0 one value (they compare equal as logits). Every real logit,
// -inf included, has a key of at least 0x007FFFFF.
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

// Walks a row of V logits spread over the CTA: fs(x) for the elements before
// the first 16-byte boundary and after the last one, fv(v) for each 16-byte
// vector in between (four loads in flight per thread). A thread sees at most
// V / blockDim + 16 elements.
template <int ES, typename FV, typename FS>
__device__ __forceinline__ void sweep_vec(const uint8_t* row, int64_t V, FV&& fv, FS&& fs)
{
    constexpr int kEPV = 16 / ES;
    constexpr int kU = 4;
    const uintptr_t p = reinterpret_cast<uintptr_t>(row);
    int64_t head = static_cast<int64_t>(((16u - static_cast<uint32_t>(p & 15u)) & 15u) / ES);
    if (head > V) head = V;
    const int64_t nvec = (V - head) / kEPV;
    const int64_t tail = head + nvec * kEPV;
    const int64_t T = blockDim.x;
    for (int64_t i = threadIdx.x; i < head; i += T) fs(load_elem<ES>(row + i * ES));
    const uint4* vp = reinterpret_cast<const uint4*>(row + head * ES);
    int64_t v = threadIdx.x;
    for (; v + (kU - 1) * T < nvec; v += kU * T) {
        uint4 u[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) u[q] = __ldg(vp + v + q * T);
#pragma unroll
        for (int q = 0; q < kU; ++q) fv(u[q]);
    }
    for (; v < nvec; v += T) fv(__ldg(vp + v));
    for (int64_t i = tail + threadIdx.x; i < V; i += T) fs(load_elem<ES>(row + i * ES));
}

// f(x) for every element of the row.
template <int ES, typename F>
__device__ __forceinline__ void sweep(const uint8_t* row, int64_t V, F&& f)
{
    sweep_vec<ES>(
        row, V,
        [&](const uint4& u) {
            float x[16 / ES];
            unpack_vec<ES>(u, x);
#pragma unroll
            for (int e = 0; e < 16 / ES; ++e) f(x[e]);
        },
        f);
}

struct Scratch {
    uint64_t wsum[kWarpsF];
    float wmax[kWarpsF];
    uint64_t tot[kDBins + 1];
    uint64_t above;
    int e;
    int lo;
    int list_n;
};

template <typename H>
__device__ __forceinline__ void zero(H* h, int n)
{
    for (int i = threadIdx.x; i < n; i += blockDim.x) h[i] = 0;
}

// Sum over the CTA (every thread gets it); integer, so the order is immaterial.
__device__ uint64_t block_sum(uint64_t x, Scratch& s)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    __syncthreads();  // s.wsum is free
    if ((threadIdx.x & 31) == 0) s.wsum[threadIdx.x >> 5] = x;
    __syncthreads();
    uint64_t t = 0;
    for (int v = 0; v < static_cast<int>(blockDim.x >> 5); ++v) t += s.wsum[v];
    return t;
}

// Appends key to the list (one shared atomic per group of lanes that append
// together); past kListCap it only counts.
__device__ __forceinline__ void append(uint32_t key, uint32_t* list, int* count)
{
    cg::coalesced_group grp = cg::coalesced_threads();
    int base = 0;
    if (grp.thread_rank() == 0) base = atomicAdd(count, static_cast<int>(grp.size()));
    base = grp.shfl(base, 0);
    const int pos = base + static_cast<int>(grp.thread_rank());
    if (pos < kListCap) list[pos] = key;
}

// Largest digit e of h[0, nb) with base + sum_{d >= e} h[d] >= target. Leaves e
// in s.e and base + sum_{d > e} h[d] in s.above. Thread t owns the bins
// [t per, (t + 1) per); a suffix scan over the threads finds the one whose
// bins hold the crossing. When even the whole histogram falls short of the
// target (fixed-point roundings of the same masses taken two ways can leave it
// a unit or so short), the lowest non-empty digit is taken, so that the
// descent ends at the smallest key it covers; s.e = -1 only when every bin is
// empty. Called by every thread of the CTA; integer sums, so the order of the
// additions is immaterial.
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
        s.lo = nb;
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
    for (int i = 0; i < per; ++i)
        if (lo + i < nb && h[lo + i] > 0) {
            atomicMin(&s.lo, lo + i);
            break;
        }
    __syncthreads();
    if (s.e < 0) {
        if (t == 0 && s.lo < nb) {
            uint64_t total = 0;
            for (int v = 0; v < nw; ++v) total += s.wsum[v];
            s.e = s.lo;
            s.above = base + total - h[s.lo];
        }
        __syncthreads();
    }
}

// Keys from a shared-memory array.
struct ListSrc {
    const uint32_t* keys;
    int n;
    template <typename F>
    __device__ __forceinline__ void each(F&& f) const
    {
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t k = keys[i];
            f(k, key_value(k));
        }
    }
};

// Keys of a whole row (read from global memory).
template <int ES>
struct RowSrc {
    const uint8_t* row;
    int64_t V;
    template <typename F>
    __device__ __forceinline__ void each(F&& f) const
    {
        sweep<ES>(row, V, [&](float x) { f(fkey(x), x); });
    }
};

// Bits of a key above an 8-bit digit at `shift` (none at the top level).
__device__ __forceinline__ uint32_t above_mask(int shift)
{
    return shift >= 24 ? 0u : (0xFFFFFFFFu << (shift + 8));
}

// Adds the per-warp histograms h[w][256] into h[0][256].
template <typename H>
__device__ __forceinline__ void fold_warps(H* h)
{
    __syncthreads();
    if (threadIdx.x < kRadixBins) {
        H x = h[threadIdx.x];
        for (int w = 1; w < kWarpsF; ++w) x += h[w * kRadixBins + threadIdx.x];
        h[threadIdx.x] = x;
    }
    __syncthreads();
}

// The k-th largest key of src (1 <= k <= the number of keys), to its top
// 8 * levels bits (the rest 0): radix select on counts.
template <typename Src>
__device__ __noinline__ uint32_t select_kth(const Src& src, uint64_t k, int levels, uint32_t* hc,
                                            Scratch& s)
{
    uint32_t* mine = hc + (threadIdx.x >> 5) * kRadixBins;
    uint32_t prefix = 0;
    uint64_t base = 0;
    for (int l = 0; l < levels; ++l) {
        const int shift = 24 - 8 * l;
        const uint32_t hi = above_mask(shift);
        __syncthreads();  // the previous level's histogram has been read
        zero(hc, kWarpsF * kRadixBins);
        __syncthreads();
        src.each([&](uint32_t key, float) {
            if ((key & hi) == prefix) atomicAdd(&mine[(key >> shift) & 0xFFu], 1u);
        });
        fold_warps(hc);
        crossing(hc, kRadixBins, base, k, s);
        const int d = s.e < 0 ? 0 : s.e;
        base = s.above;
        prefix |= static_cast<uint32_t>(d) << shift;
    }
    return prefix;
}

// Sum of the masses of src's keys >= tau.
template <typename Src>
__device__ __noinline__ uint64_t mass_ge(const Src& src, uint32_t tau, float c, float mref,
                                         Scratch& s)
{
    uint64_t acc = 0;
    src.each([&](uint32_t key, float x) {
        if (key >= tau) acc += mass_of(x, c, mref);
    });
    return block_sum(acc, s);
}

// Largest key v of src with base + (mass of src's keys >= v) >= target, by
// radix descent on masses; *kept = base + the mass of src's keys >= v.
template <typename Src>
__device__ __noinline__ uint32_t select_mass(const Src& src, uint64_t base, uint64_t target,
                                             float c, float mref, uint64_t* hm, Scratch& s,
                                             uint64_t* kept)
{
    unsigned long long* mine =
        reinterpret_cast<unsigned long long*>(hm + (threadIdx.x >> 5) * kRadixBins);
    uint32_t prefix = 0;
    int d = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        const uint32_t hi = above_mask(shift);
        __syncthreads();
        zero(hm, kWarpsF * kRadixBins);
        __syncthreads();
        src.each([&](uint32_t key, float x) {
            if ((key & hi) == prefix) {
                const uint64_t w = mass_of(x, c, mref);
                if (w) atomicAdd(&mine[(key >> shift) & 0xFFu], static_cast<unsigned long long>(w));
            }
        });
        fold_warps(hm);
        crossing(hm, kRadixBins, base, target, s);
        d = s.e < 0 ? 0 : s.e;
        base = s.above;
        prefix |= static_cast<uint32_t>(d) << shift;
    }
    *kept = base + hm[d];
    return prefix;
}

// Totals of the per-thread bins (column j of bins[kDBins][T]) in 2^40 units:
// a bin's words hold masses 2^(x c - m + edge) 2^sc, so the total is shifted
// by 40 - sc - edge (edge = j at the first level, J0 below it). Written to
// s.tot[slot(j)]: the first level puts bin j at slot 32 - j (slot 0 holds
// the tail beyond the bins), the sub-bin levels at slot 31 - j, so that slots
// grow with the logit value.
__device__ void bin_totals(const uint32_t* bins, int sc, int J0, bool first, Scratch& s)
{
    const int T = blockDim.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int j = w; j < kDBins; j += T >> 5) {
        uint64_t x = 0;
        for (int i = lane; i < T; i += 32) x += bins[j * T + i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
        if (lane == 0) {
            const int sh = 40 - sc - (first ? j : J0);
            s.tot[first ? 32 - j : 31 - j] = sh >= 0 ? (x << sh) : (x >> (-sh));
        }
    }
}

// Top-p alone on one row (see the file comment). Returns false when the row
// needs the radix select over the whole row instead.
template <int ES>
__device__ __noinline__ bool topp_bins(const uint8_t* row, int64_t V, float c, float mref,
                                       float top_p, int sc, uint32_t* bins, uint32_t* list,
                                       Scratch& s, uint32_t* tau, uint64_t* kept)
{
    const int T = blockDim.x, t = threadIdx.x;
    const float scale = __int_as_float((127 + sc) << 23);  // 2^sc
    uint64_t* hm = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(bins) + kCandBytes +
                                               kCountBytes);
    // First level: bin j = floor(log2 distance from 2^m), j < 32.
    for (int j = 0; j < kDBins; ++j) bins[j * T + t] = 0u;
    float tail = 0.f;
    sweep<ES>(row, V, [&](float x) {
        const float e = fmaf(x, c, -mref);  // log2 of the mass relative to 2^m
        if (e > -32.f) {
            int j = static_cast<int>(-e);
            j = j < 0 ? 0 : j;
            bins[j * T + t] += __float2uint_rn(ex2(e + static_cast<float>(j)) * scale);
        } else {
            tail += ex2(e);
        }
    });
    // The tail beyond 32 units: a float sum per thread, added in a fixed order.
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tail += __shfl_xor_sync(0xFFFFFFFFu, tail, off);
    __syncthreads();
    if ((t & 31) == 0) s.wsum[t >> 5] = __float2ull_rn(tail * kFix);
    __syncthreads();
    if (t == 0) {
        uint64_t z = 0;
        for (int v = 0; v < (T >> 5); ++v) z += s.wsum[v];
        s.tot[0] = z;
    }
    bin_totals(bins, sc, 0, true, s);
    __syncthreads();
    uint64_t M = 0;
    for (int j = 0; j <= kDBins; ++j) M += s.tot[j];
    const uint64_t target =
        static_cast<uint64_t>(ceil(static_cast<double>(top_p) * static_cast<double>(M)));
    crossing(s.tot, kDBins + 1, 0, target, s);
    if (s.e <= 0) return false;  // the crossing lies in the tail
    const int J0 = kDBins - s.e;
    uint64_t above = s.above;
    int chosen[kRefine];
    for (int L = 1; L <= kRefine; ++L) {
        // Read the window (bin J0, then the chosen sub-bins) into the list and,
        // in case it does not fit, into the next level's sub-bins.
        __syncthreads();
        for (int j = 0; j < kDBins; ++j) bins[j * T + t] = 0u;
        if (t == 0) s.list_n = 0;
        __syncthreads();
        sweep<ES>(row, V, [&](float x) {
            const float e = fmaf(x, c, -mref);
            if (!(e > -32.f)) return;
            int j = static_cast<int>(-e);
            j = j < 0 ? 0 : j;
            if (j != J0) return;
            // Base-32 digits of the distance's fraction u = -e - J0 (exact
            // float steps: scalings by 32 and subtractions of integers).
            float y = -e - static_cast<float>(J0);
            int idx = 0;
            for (int l = 1; l <= L; ++l) {
                y *= 32.f;
                int dl = static_cast<int>(y);
                dl = dl < 0 ? 0 : (dl > kDBins - 1 ? kDBins - 1 : dl);
                if (l == L) {
                    idx = dl;
                } else {
                    if (dl != chosen[l - 1]) return;
                    y -= static_cast<float>(dl);
                }
            }
            append(fkey(x), list, &s.list_n);
            bins[idx * T + t] += __float2uint_rn(ex2(e + static_cast<float>(J0)) * scale);
        });
        __syncthreads();
        const int n = s.list_n;
        if (n <= kListCap) {
            __syncthreads();  // every thread has read n before the bins are reused
            *tau = select_mass(ListSrc{list, n}, above, target, c, mref, hm, s, kept);
            return true;
        }
        if (L == kRefine) break;
        bin_totals(bins, sc, J0, false, s);
        __syncthreads();
        crossing(s.tot, kDBins, above, target, s);
        if (s.e < 0) return false;
        chosen[L - 1] = kDBins - 1 - s.e;
        above = s.above;
    }
    return false;
}

// The radix select over the whole row (rare: see the file comment).
template <int ES>
__device__ __noinline__ void row_select(const uint8_t* row, int64_t V, bool tk, uint64_t k,
                                        bool tp, float top_p, float c, float mref, uint32_t* hc,
                                        uint64_t* hm, Scratch& s, uint32_t* tau, uint64_t* kept)
{
    const RowSrc<ES> R{row, V};
    uint32_t t = 0;
    uint64_t m;
    if (tk) {
        t = select_kth(R, k, 4, hc, s);
        m = mass_ge(R, t, c, mref, s);
    } else {
        m = mass_ge(R, 0u, c, mref, s);
    }
    if (tp) {
        const uint64_t target =
            static_cast<uint64_t>(ceil(static_cast<double>(top_p) * static_cast<double>(m)));
        t = select_mass(R, 0, target, c, mref, hm, s, &m);
    }
    *tau = t;
    *kept = m;
}

// bf16 bits (as a float, widened) of the bf16 value whose 16-bit key is p.
__device__ __forceinline__ uint32_t bf16_bits_of_key16(uint32_t p)
{
    return (p & 0x8000u) ? (p & 0x7FFFu) : (~p & 0xFFFFu);
}

__device__ __forceinline__ unsigned ge2_mask(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    return __hge2_mask(x, y);
}

template <int ES>
__global__ void __launch_bounds__(kFilterThreads, 2) filter_kernel(const __grid_constant__ FilterArgs a)
{
    constexpr int G = groups<ES>();
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* bins = reinterpret_cast<uint32_t*>(smem);
    uint32_t* cand = bins;
    uint32_t* hc = reinterpret_cast<uint32_t*>(smem + kCandBytes);
    uint64_t* hm = reinterpret_cast<uint64_t*>(smem + kCandBytes + kCountBytes);
    uint32_t* list = reinterpret_cast<uint32_t*>(smem + kBinsBytes);
    __shared__ Scratch s;
    const Geometry& g = a.g;
    const int64_t V = g.V;
    const int T = blockDim.x, t = threadIdx.x;
    const bool tk = a.top_k > 0 && a.top_k < V;
    const bool tp = a.top_p < 1.0f;
    const uint64_t k = tk ? static_cast<uint64_t>(a.top_k) : 0;
    const bool fast_k = tk && a.top_k <= static_cast<int64_t>(G) * T;
    const float c = a.c;
    const float ninf = __uint_as_float(kF32NegInfBits);
    // Per-thread bin words add at most V / T + 16 masses of at most 2^sc (+1).
    int lg = 0;
    while ((int64_t(1) << lg) < V / T + 16) ++lg;
    const int sc = 31 - lg;
    pdl_trigger();  // the scan may launch; it waits for this grid before reading

    for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const uint8_t* row =
            r < g.rows_t ? a.target + r * V * ES : a.draft + (r - g.rows_t) * V * ES;
        __syncthreads();  // the previous row is done with shared memory

        // First read (HBM): the NaN-propagating maximum of each lane position
        // of this thread's vectors (scalar head / tail elements join group 0).
        float gm[G];
        {
            float hs = ninf;
            if constexpr (ES == 2) {
                uint32_t acc[4] = {kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair};
                sweep_vec<ES>(
                    row, V,
                    [&](const uint4& u) {
                        acc[0] = bf16x2_max_nan(acc[0], u.x);
                        acc[1] = bf16x2_max_nan(acc[1], u.y);
                        acc[2] = bf16x2_max_nan(acc[2], u.z);
                        acc[3] = bf16x2_max_nan(acc[3], u.w);
                    },
                    [&](float x) { hs = fmax_nan(hs, x); });
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    gm[2 * q] = bf16_lo(acc[q]);
                    gm[2 * q + 1] = bf16_hi(acc[q]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < G; ++q) gm[q] = ninf;
                sweep_vec<ES>(
                    row, V,
                    [&](const uint4& u) {
                        gm[0] = fmax_nan(gm[0], __uint_as_float(u.x));
                        gm[1] = fmax_nan(gm[1], __uint_as_float(u.y));
                        gm[2] = fmax_nan(gm[2], __uint_as_float(u.z));
                        gm[3] = fmax_nan(gm[3], __uint_as_float(u.w));
                    },
                    [&](float x) { hs = fmax_nan(hs, x); });
            }
            gm[0] = fmax_nan(gm[0], hs);
        }
        float mx = gm[0];
#pragma unroll
        for (int q = 1; q < G; ++q) mx = fmax_nan(mx, gm[q]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmax_nan(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if ((t & 31) == 0) s.wmax[t >> 5] = mx;
        __syncthreads();
        for (int v = 0; v < (T >> 5); ++v) mx = fmax_nan(mx, s.wmax[v]);
        // NaN anywhere makes the maximum NaN; +inf makes it +inf.
        if (!(mx > ninf) || !(mx < __uint_as_float(0x7F800000u))) {
            if (t == 0) a.rows[r] = FiltRow{0.f, 0.f, 0.f, kFlagNonFinite};
            continue;
        }
        const float mref = ceilf(mx * c);

        uint32_t tau = 0;  // threshold key
        uint64_t kept = 0;
        bool done = false;
        if (fast_k) {
            // The group maxima are G T disjoint elements (an empty group's -inf
            // only lowers the bound), so at least k elements are >= the k-th
            // largest of them; to 16 bits it is a lower bound on the k-th
            // largest logit.
#pragma unroll
            for (int q = 0; q < G; ++q) cand[G * t + q] = fkey(gm[q]);
            if (t == 0) s.list_n = 0;
            __syncthreads();
            const uint32_t p16 = select_kth(ListSrc{cand, G * T}, k, 2, hc, s) >> 16;
            // The 16-bit prefix of -inf's key (0x007FFFFF) or below: no bound.
            const bool open = p16 <= 0x007Fu;
            const float bound = open ? ninf : key_value(p16 << 16);
            const uint32_t b16 = open ? 0xFF80u : bf16_bits_of_key16(p16);
            const uint32_t b2 = b16 | (b16 << 16);
            // Second read: every element >= the bound joins the list.
            sweep_vec<ES>(
                row, V,
                [&](const uint4& u) {
                    bool any;
                    if constexpr (ES == 2) {
                        any = (ge2_mask(u.x, b2) | ge2_mask(u.y, b2) | ge2_mask(u.z, b2) |
                               ge2_mask(u.w, b2)) != 0u;
                    } else {
                        any = (__uint_as_float(u.x) >= bound) | (__uint_as_float(u.y) >= bound) |
                              (__uint_as_float(u.z) >= bound) | (__uint_as_float(u.w) >= bound);
                    }
                    if (any) {
                        float x[16 / ES];
                        unpack_vec<ES>(u, x);
#pragma unroll
                        for (int e = 0; e < 16 / ES; ++e)
                            if (x[e] >= bound) append(fkey(x[e]), list, &s.list_n);
                    }
                },
                [&](float x) {
                    if (x >= bound) append(fkey(x), list, &s.list_n);
                });
            __syncthreads();
            const int n = s.list_n;
            if (n <= kListCap) {
                const ListSrc L{list, n};
                tau = select_kth(L, k, 4, hc, s);
                kept = mass_ge(L, tau, c, mref, s);
                if (tp) {
                    const uint64_t target = static_cast<uint64_t>(
                        ceil(static_cast<double>(a.top_p) * static_cast<double>(kept)));
                    tau = select_mass(L, 0, target, c, mref, hm, s, &kept);
                }
                done = true;
            }
        } else if (tp && !tk) {
            done = topp_bins<ES>(row, V, c, mref, a.top_p, sc, bins, list, s, &tau, &kept);
        }
        if (!done) row_select<ES>(row, V, tk, k, tp, a.top_p, c, mref, hc, hm, s, &tau, &kept);
        if (t == 0) {
            const float thr = tau == 0u ? ninf : key_value(tau);
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
