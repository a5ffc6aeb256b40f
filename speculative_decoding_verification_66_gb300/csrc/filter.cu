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
// This kernel takes top-k up to 64 (with or without top-p) for both dtypes,
// and every cut of float32 rows; bfloat16 rows cut by top-p alone or by top-k
// above 64 go to the value-count kernel (hist.cu).
//
// Design: one CTA per row (a persistent grid walks the rows). The exact
// thresholds come from a radix select over 32-bit order-preserving keys of
// the widened logits, 8 bits per level, with shared-memory histograms of
// counts (top-k) and masses (top-p), one copy per warp so that lanes of
// different warps never contend. Run over a whole row, that select would cost
// some twenty instructions and a contended atomic per element -- several
// times the HBM budget -- so it runs on a short list of candidates instead:
//  * first read (HBM): each thread keeps, per lane position of its 16-byte
//    vectors (a group), the maximum and the second largest value (packed
//    NaN-propagating max and min, about 1.5 instructions per bf16 element),
//    which gives the row maximum, the NaN / +inf check and 2048 (bf16) or
//    1024 (fp32) group maxima of disjoint groups.
//  * top-k (with or without top-p): the k-th largest thread maximum (k up to
//    64: the CTA sorts the 256 of them) or group maximum (larger k, float32
//    rows: a radix select) bounds the k-th largest logit from below. A group
//    whose second value is below the bound holds at most one element above
//    it, its maximum, which joins the list; the few thread shares with a
//    group of two or more are read again (from L2), or, when more than 16
//    are, the whole row with a packed compare. The list then holds the whole
//    top-k set (about k keys), and the cuts are resolved on it: one warp sorts
//    lists of up to 128 keys, the CTA ranks lists of up to 512, a radix select
//    takes longer ones.
//  * top-p alone (float32 rows): the second read adds each element's mass
//    into per-thread private bins (no atomics) by its log2 distance from the
//    row maximum, 32 bins of one unit; the bin where the running mass from the
//    top reaches top_p times the row mass is read again into the list, or,
//    when it holds too many elements, split into 32 sub-bins the same way, up
//    to three times.
//  * anything else (a list that overflows, a crossing in the bins' far tail)
//    runs the radix select over the whole row.
// Sweeps after the first read the row again, normally from L2 (four CTAs per
// SM keep about 600 rows, some 150 MB of bf16 rows of 128K tokens, in flight,
// so a share read again may also come from HBM).
//
// Masses are integers, so every sum -- and every decision -- is the same on
// every run: a list element's mass is its 2^(x c - m) (m the ceiling of
// max x c) scaled by 2^40 and rounded; a bin adds per-thread 32-bit sums of
// its elements' masses relative to the bin's reference power of two, scaled by
// 2^SC with SC chosen so that a thread's sum cannot overflow, and rescaled by
// a shift.
// The roundings (below 2^-22 of each element's mass) and the SFU exponential
// (a few ulp per term) move a top-p boundary by well under 1e-5 of the mass.
#include <cooperative_groups.h>

#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_stages.h"

namespace sv {
namespace {

namespace cg = cooperative_groups;

constexpr int kFilterThreads = 256;
constexpr int kWarpsF = kFilterThreads / 32;
constexpr int kCand = 8;                             // group maxima per thread (bf16; fp32: 4)
constexpr int kListCap = 4096;                       // list entries (keys)
constexpr int kDBins = 32;                           // log2-distance bins per level
constexpr int kRefine = 3;                           // sub-bin levels after the first
constexpr int kRadixBins = 256;                      // 8-bit digits
constexpr int kMaxShares = 16;                       // thread shares read again (else the whole row)
constexpr int kSortK = 64;                           // k up to which the thread maxima give the bound
constexpr float kFix = 1099511627776.0f;             // 2^40

// Dynamic shared memory: the per-thread bins [kDBins][kFilterThreads]; during
// the reads that use it, the same 32 KB hold the bulk-copy ring, and in every
// select the candidate keys (first 4 KB), the per-warp counts (next 8 KB) and
// the per-warp masses (16 KB). Then the list.
constexpr size_t kBinsBytes = sizeof(uint32_t) * kDBins * kFilterThreads;
constexpr size_t kCandBytes = sizeof(uint32_t) * kCand * kFilterThreads;
constexpr size_t kCountBytes = sizeof(uint32_t) * kWarpsF * kRadixBins;
constexpr size_t kMassBytes = sizeof(uint64_t) * kWarpsF * kRadixBins;
constexpr size_t kListBytes = sizeof(uint32_t) * kListCap;
constexpr size_t kFilterSmem = kBinsBytes + kListBytes;
static_assert(kCandBytes + kCountBytes + kMassBytes <= kBinsBytes, "select scratch fits the bins");

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
    int inc_n;
    int check;  // kFlagIndex when a device-side index check failed on this row
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

// Rows whose length is a whole number of 16-byte vectors stream through a
// ring of bulk copies: thread 0 issues the copies, every thread waits on the
// stage's mbarrier, reads its vectors from shared memory, and the CTA barrier
// after each tile frees the stage for the copy nst tiles ahead. The first read
// of a row has all 48 KB of shared memory free and runs three stages; later
// reads run two, in whichever region they leave free.
constexpr int kTileBytes = 16384;
constexpr int kStages = 2;
constexpr int kFirstStages = 3;
static_assert(kStages * kTileBytes <= static_cast<int>(kBinsBytes), "ring fits the bins");
static_assert(kFirstStages * kTileBytes <= static_cast<int>(kBinsBytes + kListBytes),
              "first-read ring fits shared memory");

struct Ring {
    uint64_t* bar;   // [kFirstStages] mbarriers
    uint8_t* buf;    // nst tiles
    uint32_t phase;  // bit s: parity of the next wait on stage s
    int tile;        // bytes per stage (a multiple of 16)
    int nst;         // stages in use (kStages, or kFirstStages for a row's first read)
};

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// fv(v) for every 16-byte vector of a row of `bytes` bytes (a multiple of 16,
// 16-byte aligned). False if a copy did not land within the wait limit; the
// copies still pending have then been waited for (bounded) and the ring must
// not be used again.
template <typename FV>
__device__ bool ring_sweep(Ring& rg, const uint8_t* row, int64_t bytes, FV&& fv)
{
    const int t = threadIdx.x, T = blockDim.x;
    const int64_t tb = rg.tile;
    const int64_t ntiles = (bytes + tb - 1) / tb;
    auto tile_bytes = [&](int64_t i) {
        const int64_t n = bytes - i * tb;
        return static_cast<uint32_t>(n < tb ? n : tb);
    };
    const int nst = rg.nst;
    auto issue = [&](int64_t i) {
        const int st = static_cast<int>(i % nst);
        mbar_arrive_expect_tx(&rg.bar[st], tile_bytes(i));
        bulk_copy_g2s(rg.buf + st * tb, row + i * tb, tile_bytes(i), &rg.bar[st]);
    };
    if (t == 0) {
        fence_proxy_async();  // earlier generic accesses to the buffer come first
        for (int64_t i = 0; i < ntiles && i < nst; ++i) issue(i);
    }
    for (int64_t i = 0; i < ntiles; ++i) {
        const int st = static_cast<int>(i % nst);
        bool ok = mbar_wait_bounded(&rg.bar[st], (rg.phase >> st) & 1u, nullptr);
        rg.phase ^= 1u << st;
        if (ok) {
            const uint8_t* base = rg.buf + st * tb;
            const int nvec = static_cast<int>(tile_bytes(i) / 16);
            for (int v = t; v < nvec; v += T) fv(ld_shared_v4(base + 16 * v));
        }
        if (!__syncthreads_and(ok)) {
            // Let the copies still in flight land before giving up.
            if (!ok) mbar_wait_bounded(&rg.bar[st], ((rg.phase >> st) & 1u) ^ 1u, nullptr);
            for (int j = 1; j < nst && i + j < ntiles; ++j) {
                const int sn = static_cast<int>((i + j) % nst);
                mbar_wait_bounded(&rg.bar[sn], (rg.phase >> sn) & 1u, nullptr);
            }
            return false;
        }
        if (t == 0 && i + nst < ntiles) issue(i + nst);
    }
    return true;
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

// Warp-aggregated histogram updates for a warp whose 32 lanes all call them
// (digit -1: nothing to add). Lanes with the same digit form one group; its
// lowest lane adds the group's count or mass to the warp's private row, so no
// two lanes ever update one word at once (same-address shared atomics replay
// once per conflicting lane, and list keys crowd into few digits).
__device__ __forceinline__ void warp_add_count(uint32_t* mine, int digit)
{
    const unsigned m = __match_any_sync(0xFFFFFFFFu, digit);
    if (digit >= 0 && static_cast<int>(threadIdx.x & 31) == __ffs(m) - 1) mine[digit] += __popc(m);
}

// Masses below 2^55: the low 23 and the high bits are summed separately as
// 32-bit words (32 lanes cannot overflow either), then recombined exactly.
__device__ __forceinline__ void warp_add_mass(uint64_t* mine, int digit, uint64_t w)
{
    const unsigned m = __match_any_sync(0xFFFFFFFFu, digit);
    const uint32_t lo = __reduce_add_sync(m, static_cast<uint32_t>(w & 0x7FFFFFu));
    const uint32_t hi = __reduce_add_sync(m, static_cast<uint32_t>(w >> 23));
    if (digit >= 0 && static_cast<int>(threadIdx.x & 31) == __ffs(m) - 1)
        mine[digit] += (static_cast<uint64_t>(hi) << 23) + lo;
}

// The k-th largest of n keys in shared memory (1 <= k <= n), to its top
// 8 * levels bits: radix select with warp-aggregated histograms.
__device__ __noinline__ uint32_t list_select_kth(const uint32_t* keys, int n, uint64_t k, int levels,
                                                 uint32_t* hc, Scratch& s)
{
    uint32_t* mine = hc + (threadIdx.x >> 5) * kRadixBins;
    uint32_t prefix = 0;
    uint64_t base = 0;
    for (int l = 0; l < levels; ++l) {
        const int shift = 24 - 8 * l;
        const uint32_t hi = above_mask(shift);
        __syncthreads();
        zero(hc, kWarpsF * kRadixBins);
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += blockDim.x) {
            const int i = i0 + static_cast<int>(threadIdx.x);
            const uint32_t key = i < n ? keys[i] : 0u;
            const bool in = i < n && (key & hi) == prefix;
            warp_add_count(mine, in ? static_cast<int>((key >> shift) & 0xFFu) : -1);
        }
        fold_warps(hc);
        crossing(hc, kRadixBins, base, k, s);
        const int d = s.e < 0 ? 0 : s.e;
        base = s.above;
        prefix |= static_cast<uint32_t>(d) << shift;
    }
    return prefix;
}

// select_mass over n keys in shared memory, with warp-aggregated histograms.
__device__ __noinline__ uint32_t list_select_mass(const uint32_t* keys, int n, uint64_t base,
                                                  uint64_t target, float c, float mref,
                                                  uint64_t* hm, Scratch& s, uint64_t* kept)
{
    uint64_t* mine = hm + (threadIdx.x >> 5) * kRadixBins;
    uint32_t prefix = 0;
    int d = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        const uint32_t hi = above_mask(shift);
        __syncthreads();
        zero(hm, kWarpsF * kRadixBins);
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += blockDim.x) {
            const int i = i0 + static_cast<int>(threadIdx.x);
            const uint32_t key = i < n ? keys[i] : 0u;
            const bool in = i < n && (key & hi) == prefix;
            const uint64_t w = in ? mass_of(key_value(key), c, mref) : 0u;
            warp_add_mass(mine, in ? static_cast<int>((key >> shift) & 0xFFu) : -1, w);
        }
        fold_warps(hm);
        crossing(hm, kRadixBins, base, target, s);
        d = s.e < 0 ? 0 : s.e;
        base = s.above;
        prefix |= static_cast<uint32_t>(d) << shift;
    }
    *kept = base + hm[d];
    return prefix;
}

// Sorts 32 P keys held P per lane (key r of lane l is element l P + r) into
// descending order across the warp: a bitonic network, compare-exchanges in
// registers for partners in the same lane and by shuffles otherwise.
template <int P>
__device__ __forceinline__ void warp_sort_desc(uint32_t (&v)[P], int lane)
{
    constexpr int N = 32 * P;
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < P) {
#pragma unroll
                for (int r = 0; r < P; ++r) {
                    if (r & stride) continue;
                    const int e = lane * P + r;
                    const uint32_t hi = max(v[r], v[r | stride]), lo = min(v[r], v[r | stride]);
                    const bool desc = (e & size) == 0;
                    v[r] = desc ? hi : lo;
                    v[r | stride] = desc ? lo : hi;
                }
            } else {
                const int lm = stride / P;
                const bool lower = (lane & lm) == 0;
#pragma unroll
                for (int r = 0; r < P; ++r) {
                    const int e = lane * P + r;
                    const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, v[r], lm);
                    const bool desc = (e & size) == 0;
                    v[r] = (lower == desc) ? max(v[r], o) : min(v[r], o);
                }
            }
        }
    }
}

// Top-k then top-p on a list of n <= kSmallList keys by one warp, without
// block barriers. The warp sorts the keys in descending order (a bitonic
// network over P keys per lane, lane l holding positions l*P .. l*P+P-1, the
// padding keys 0 sinking below every real key); a key's rank window is then
// its position, and masses follow from the sorted keys. The k-th largest key
// tau_k sits at position k-1; the top-p threshold is the key at the first
// position whose inclusive mass prefix reaches ceil(top_p * mass(tau_k)) —
// the largest key whose upper-set mass reaches it, since every earlier tie
// group ends before that position. Every lane returns the results.
constexpr int kSmallList = 128;

template <int P>
__device__ __forceinline__ void small_select_p(const uint32_t* keys, int n, bool tk, uint64_t k, bool tp,
                                               float top_p, float c, float mref, uint32_t* tau_out,
                                               uint64_t* kept_out)
{
    const int lane = threadIdx.x & 31;
    uint32_t v[P];
#pragma unroll
    for (int r = 0; r < P; ++r) {
        const int i = lane * P + r;
        v[r] = i < n ? keys[i] : 0u;
    }
    warp_sort_desc<P>(v, lane);
    uint64_t w[P];
#pragma unroll
    for (int r = 0; r < P; ++r) w[r] = lane * P + r < n ? mass_of(key_value(v[r]), c, mref) : 0u;
    // The key at sorted position pos (0 <= pos < 32 P), broadcast from its lane.
    auto at = [&](int pos) {
        uint32_t mine = v[0];
#pragma unroll
        for (int r = 1; r < P; ++r)
            if (pos % P == r) mine = v[r];
        return __shfl_sync(0xFFFFFFFFu, mine, pos / P);
    };
    // Sum of the masses of the real keys >= x, over the warp.
    auto mass_ge = [&](uint32_t x) {
        uint64_t acc = 0;
#pragma unroll
        for (int r = 0; r < P; ++r)
            if (lane * P + r < n && v[r] >= x) acc += w[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
        return acc;
    };
    uint32_t tau;
    if (tk)
        tau = (k >= 1 && k <= static_cast<uint64_t>(n)) ? at(static_cast<int>(k) - 1) : 0u;
    else
        tau = n > 0 ? at(n - 1) : 0xFFFFFFFFu;
    const uint64_t mass_k = mass_ge(tau);
    uint64_t kept = mass_k;
    if (tp) {
        const uint64_t target =
            static_cast<uint64_t>(ceil(static_cast<double>(top_p) * static_cast<double>(mass_k)));
        uint64_t run = 0;
#pragma unroll
        for (int r = 0; r < P; ++r) run += w[r];
        // Exclusive prefix of the lane totals.
        uint64_t inc = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
            if (lane >= off) inc += o;
        }
        run = inc - run;
        int first = -1;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            run += w[r];
            if (first < 0 && lane * P + r < n && run >= target) first = r;
        }
        // No hit, or a hit on key 0 (no logit has it), leaves (0, 0).
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, first >= 0);
        tau = 0u;
        kept = 0u;
        if (hit != 0u) {
            const int src = __ffs(hit) - 1;
            const int r0 = __shfl_sync(0xFFFFFFFFu, first, src);
            tau = at(src * P + r0);
            if (tau != 0u) kept = mass_ge(tau);
        }
    }
    *tau_out = tau;
    *kept_out = kept;
}

__device__ __noinline__ void small_select(const uint32_t* keys, int n, bool tk, uint64_t k, bool tp,
                                          float top_p, float c, float mref, uint32_t* tau_out,
                                          uint64_t* kept_out)
{
    if (n <= 32)
        small_select_p<1>(keys, n, tk, k, tp, top_p, c, mref, tau_out, kept_out);
    else if (n <= 64)
        small_select_p<2>(keys, n, tk, k, tp, top_p, c, mref, tau_out, kept_out);
    else
        small_select_p<4>(keys, n, tk, k, tp, top_p, c, mref, tau_out, kept_out);
}

// small_select for lists of up to kMidList keys by the whole CTA: each thread
// ranks its elements (i = t + j blockDim) against the whole list; the k-th
// largest key, the top-k mass and the top-p threshold then take a few block
// reductions. Every thread returns the results.
constexpr int kMidList = 512;

__device__ __noinline__ void mid_select(const uint32_t* keys, int n, uint64_t k, bool tp, float top_p,
                                        float c, float mref, uint64_t* w, Scratch& s,
                                        uint32_t* tau_out, uint64_t* kept_out)
{
    constexpr int kPer = kMidList / kFilterThreads;
    const int t = threadIdx.x, T = blockDim.x;
    for (int i = t; i < n; i += T) w[i] = mass_of(key_value(keys[i]), c, mref);
    if (t == 0) {
        s.lo = 0;
        s.e = 0;
    }
    __syncthreads();
    uint32_t kk[kPer];
    int gt[kPer], ge[kPer];
    uint64_t up[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        kk[q] = t + q * T < n ? keys[t + q * T] : 0u;
        gt[q] = ge[q] = 0;
        up[q] = 0;
    }
    for (int j = 0; j < n; ++j) {
        const uint32_t kj = keys[j];
        const uint64_t wj = w[j];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            gt[q] += kj > kk[q];
            ge[q] += kj >= kk[q];
            up[q] += kj >= kk[q] ? wj : 0u;
        }
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q)
        if (t + q * T < n && static_cast<uint64_t>(gt[q]) < k && static_cast<uint64_t>(ge[q]) >= k)
            s.lo = static_cast<int>(kk[q]);  // every such element holds the same key
    __syncthreads();
    uint32_t tau = static_cast<uint32_t>(s.lo);
    uint64_t mk = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q)
        if (t + q * T < n && kk[q] >= tau) mk += w[t + q * T];
    const uint64_t mass_k = block_sum(mk, s);
    uint64_t kept = mass_k;
    if (tp) {
        const uint64_t target =
            static_cast<uint64_t>(ceil(static_cast<double>(top_p) * static_cast<double>(mass_k)));
        uint32_t best = 0u;
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (t + q * T < n && up[q] >= target && kk[q] > best) best = kk[q];
        atomicMax(reinterpret_cast<unsigned int*>(&s.e), best);
        __syncthreads();
        tau = static_cast<uint32_t>(s.e);
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if (t + q * T < n && kk[q] == tau) s.above = up[q];  // equal keys, equal sums
        __syncthreads();
        kept = s.above;
    }
    *tau_out = tau;
    *kept_out = kept;
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

// Conversions by float addition instead of float <-> integer conversions
// (those issue at a quarter of the rate; these are one add and one integer
// subtract): adding 1.5 * 2^23 to a float of magnitude below 2^22 rounds it to
// an integer held in the low mantissa bits.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;

// First-level bin of a log2 mass e (e <= 0 up to rounding): j = round(-e),
// r = j as a float. The bin's masses 2^e lie within a factor 2^(1/2) of 2^-j.
struct DBin {
    int j;
    float r;
};
__device__ __forceinline__ DBin dbin(float e)
{
    const float y = kMagic - e;
    int j = static_cast<int>(__float_as_uint(y) - kMagicBits);
    j = j < 0 ? 0 : (j > kDBins - 1 ? kDBins - 1 : j);
    return DBin{j, static_cast<float>(y - kMagic)};
}

// round(m * scale) for 0 <= m * scale < 2^22.
__device__ __forceinline__ uint32_t to_fixed(float m, float scale)
{
    return __float_as_uint(fmaf(m, scale, 8388608.0f)) - 0x4B000000u;
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

// Top-p alone on one row (see the file comment). Returns 1 when done, 0 when
// the row needs the radix select over the whole row instead, -1 when a bulk
// copy did not arrive in time. Rows of whole 16-byte vectors stream through
// the ring, placed in whichever region the sweep leaves free: the list while
// per-thread bins are being filled, the bins while the list is.
template <int ES>
__device__ __noinline__ int topp_bins(const uint8_t* row, int64_t V, float c, float mref,
                                      float top_p, int sc, uint32_t* bins, uint32_t* list,
                                      Scratch& s, Ring& rg, bool use_ring, uint32_t* tau,
                                      uint64_t* kept)
{
    const int T = blockDim.x, t = threadIdx.x;
    const float scale = __int_as_float((127 + sc) << 23);  // 2^sc
    uint64_t* hm = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(bins) + kCandBytes +
                                               kCountBytes);
    // f(x) for every element; false if a copy did not land.
    auto each = [&](bool ring_in_list, auto&& f) -> bool {
        if (!use_ring) {
            sweep<ES>(row, V, f);
            return true;
        }
        rg.buf = ring_in_list ? reinterpret_cast<uint8_t*>(list) : reinterpret_cast<uint8_t*>(bins);
        rg.tile = ring_in_list ? static_cast<int>(kListBytes / kStages) : kTileBytes;
        rg.nst = kStages;
        return ring_sweep(rg, row, V * ES, [&](const uint4& u) {
            float x[16 / ES];
            unpack_vec<ES>(u, x);
#pragma unroll
            for (int e = 0; e < 16 / ES; ++e) f(x[e]);
        });
    };
    // First level: bin j = round(log2 distance from 2^m), j < 32.
    for (int j = 0; j < kDBins; ++j) bins[j * T + t] = 0u;
    float tail = 0.f;
    __syncthreads();  // the list region is free for the ring
    if (!each(true, [&](float x) {
        const float e = fmaf(x, c, -mref);  // log2 of the mass relative to 2^m
        if (e > -31.5f) {
            const DBin b = dbin(e);
            bins[b.j * T + t] += to_fixed(ex2(e + b.r), scale);
        } else {
            tail += ex2(e);
        }
    }))
        return -1;
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
    if (s.e <= 0) return 0;  // the crossing lies in the tail
    const int J0 = kDBins - s.e;
    uint64_t above = s.above;
    // The window (bin J0, then sub-bins of it) spans log2 distances
    // [J0 - 1/2 + off, J0 - 1/2 + off + width); each of its elements has a
    // mass of at least 2^(40 - (far edge)) in 2^40 units, so the window's mass
    // bounds its count.
    uint64_t wmass = s.tot[s.e];
    double off = 0.0, width = 1.0;
    int chosen[kRefine];
    for (int L = 0; L <= kRefine; ++L) {
        const double ub =
            static_cast<double>(wmass) / exp2(40.0 - (J0 - 0.5 + off + width)) * 1.001 + 16.0;
        const bool collect = ub <= kListCap || L == kRefine;
        // Read the window: into the list when it fits, else into the next
        // level's 32 sub-bins.
        __syncthreads();
        if (!collect)
            for (int j = 0; j < kDBins; ++j) bins[j * T + t] = 0u;
        if (t == 0) s.list_n = 0;
        __syncthreads();
        if (!each(!collect, [&](float x) {
            const float e = fmaf(x, c, -mref);
            if (!(e > -31.5f)) return;
            const DBin b = dbin(e);
            if (b.j != J0) return;
            // Base-32 digits of the distance's offset in the bin, y = -e - J0
            // + 1/2 in [0, 1] (monotone float steps: scalings by 32 and
            // subtractions of integers).
            float y = (-e - b.r) + 0.5f;
            for (int l = 0; l < L; ++l) {
                y *= 32.f;
                int dl = static_cast<int>(y);
                dl = dl < 0 ? 0 : (dl > kDBins - 1 ? kDBins - 1 : dl);
                if (dl != chosen[l]) return;
                y -= static_cast<float>(dl);
            }
            if (collect) {
                append(fkey(x), list, &s.list_n);
            } else {
                int idx = static_cast<int>(y * 32.f);
                idx = idx < 0 ? 0 : (idx > kDBins - 1 ? kDBins - 1 : idx);
                bins[idx * T + t] += to_fixed(ex2(e + b.r), scale);
            }
        }))
            return -1;
        __syncthreads();
        if (collect) {
            const int n = s.list_n;
            if (n > kListCap) return 0;
            __syncthreads();  // every thread has read n before the bins are reused
            *tau = list_select_mass(list, n, above, target, c, mref, hm, s, kept);
            return 1;
        }
        bin_totals(bins, sc, J0, false, s);
        __syncthreads();
        crossing(s.tot, kDBins, above, target, s);
        if (s.e < 0) return 0;
        chosen[L] = kDBins - 1 - s.e;
        above = s.above;
        wmass = s.tot[s.e];
        off += chosen[L] * (width / kDBins);
        width /= kDBins;
    }
    return 0;
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

// The 16 bits of the bf16 value whose 16-bit key is p.
__device__ __forceinline__ uint32_t bf16_bits_of_key16(uint32_t p)
{
    return (p & 0x8000u) ? (p & 0x7FFFu) : (~p & 0xFFFFu);
}

// Packed x >= y on both bf16 halves: 0xFFFF per half where it holds.
__device__ __forceinline__ unsigned ge2_mask(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    return __hge2_mask(x, y);
}

// Lane-wise minimum of two packed bfloat16 pairs.
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Appends every element >= lk (by key) of the shares of threads inc[0 .. ninc)
// of the row: a share is the head / tail indices and 16-byte vectors
// congruent to its thread index modulo the block size, as the reads give them
// out. The CTA reads the shares' vectors together, one vector per thread per
// round, the loads of a round issued before any is used.
template <int ES>
__device__ __forceinline__ void reread_shares(const uint8_t* row, int64_t V, const int* inc, int ninc,
                                           uint32_t lk, uint32_t* list, int* count)
{
    constexpr int kEPV = 16 / ES;
    constexpr int kU = 4;
    const uintptr_t p = reinterpret_cast<uintptr_t>(row);
    int64_t head = static_cast<int64_t>(((16u - static_cast<uint32_t>(p & 15u)) & 15u) / ES);
    if (head > V) head = V;
    const int64_t nvec = (V - head) / kEPV;
    const int64_t tail = head + nvec * kEPV;
    const int64_t T = blockDim.x;
    if (threadIdx.x < ninc) {
        const int tt = inc[threadIdx.x];
        if (tt < head) {
            const uint32_t key = fkey(load_elem<ES>(row + tt * ES));
            if (key >= lk) append(key, list, count);
        }
        if (tail + tt < V) {
            const uint32_t key = fkey(load_elem<ES>(row + (tail + tt) * ES));
            if (key >= lk) append(key, list, count);
        }
    }
    const uint4* vp = reinterpret_cast<const uint4*>(row + head * ES);
    const int64_t per = (nvec + T - 1) / T;  // vectors in a share (at most)
    const int64_t items = per * ninc;
    for (int64_t i0 = threadIdx.x; i0 < items; i0 += kU * T) {
        uint4 u[kU];
        bool ok[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t i = i0 + q * T;
            const int64_t g = i < items ? inc[i / per] + (i % per) * T : nvec;
            ok[q] = g < nvec;
            if (ok[q]) u[q] = __ldg(vp + g);
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            if (!ok[q]) continue;
            float x[kEPV];
            unpack_vec<ES>(u[q], x);
#pragma unroll
            for (int e = 0; e < kEPV; ++e) {
                const uint32_t key = fkey(x[e]);
                if (key >= lk) append(key, list, count);
            }
        }
    }
}

__device__ __forceinline__ void fail_rows(const FilterArgs& a, int64_t r)
{
    if (threadIdx.x == 0)
        for (int64_t q = r; q < a.g.rows; q += gridDim.x) a.rows[q] = FiltRow{0.f, 0.f, 0.f, kFlagTimeout};
}

template <int ES>
__global__ void __launch_bounds__(kFilterThreads, 4) filter_kernel(const __grid_constant__ FilterArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* bins = reinterpret_cast<uint32_t*>(smem);
    uint32_t* cand = bins;
    uint32_t* hc = reinterpret_cast<uint32_t*>(smem + kCandBytes);
    uint64_t* hm = reinterpret_cast<uint64_t*>(smem + kCandBytes + kCountBytes);
    uint32_t* list = reinterpret_cast<uint32_t*>(smem + kBinsBytes);
    __shared__ Scratch s;
    __shared__ __align__(8) uint64_t ring_bar[kFirstStages];
    const Geometry& g = a.g;
    const int64_t V = g.V;
    const int T = blockDim.x, t = threadIdx.x;
    // Whole 16-byte vectors per row: every row starts 16-byte aligned.
    const bool use_ring = (V * ES) % 16 == 0;
    Ring rg{ring_bar, smem, 0u, kTileBytes, kStages};
    if (t == 0) {
        for (int i = 0; i < kFirstStages; ++i) mbar_init(&ring_bar[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const bool tk = a.top_k > 0 && a.top_k < V;
    const bool tp = a.top_p < 1.0f;
    const uint64_t k = tk ? static_cast<uint64_t>(a.top_k) : 0;
    constexpr int G = 16 / ES;  // groups per thread: the lane positions of a 16-byte vector
    const bool fast_k = tk && a.top_k <= static_cast<int64_t>(G) * T;
    const float c = a.c;
    const float ninf = __uint_as_float(kF32NegInfBits);
    // Per-thread bin words add at most V / T + 16 masses of at most
    // 2^(sc + 1/2) (+1/2).
    int lg = 0;
    while ((int64_t(1) << lg) < V / T + 16) ++lg;
    // One bit of headroom for masses up to 2^(1/2) of a bin's reference, and
    // at most 22 bits so that to_fixed stays exact.
    const int sc = 30 - lg < 22 ? 30 - lg : 22;
    pdl_trigger();  // the scan may launch; it waits for this grid before reading
    if (a.gate != nullptr) {
        // Test hook: hold every copy until *gate != 0, bounded like every
        // other wait. Nothing sets it in the tests that use it: the CTA then
        // marks its rows as timed out and returns, with no copy issued.
        if (t == 0) {
            s.list_n = 0;
            const volatile int32_t* gate = a.gate;
            const long long t0 = clock64();
            while (*gate == 0) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    s.list_n = 1;
                    break;
                }
                __nanosleep(1000);
            }
        }
        __syncthreads();
        if (s.list_n != 0) {
            fail_rows(a, blockIdx.x);
            return;
        }
    }

    for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const uint8_t* row =
            r < g.rows_t ? a.target + r * V * ES : a.draft + (r - g.rows_t) * V * ES;
        if (t == 0) s.check = 0;  // thread 0 wrote the previous row's result
        __syncthreads();  // the previous row is done with shared memory

        // First read (HBM): per lane position of this thread's vectors (a
        // group), the NaN-propagating maximum and the second largest value
        // (packed min / max, no branches). Scalar head / tail elements form
        // one more group, folded into group 0 afterwards.
        float m1[G], m2[G];
        bool landed = true;
        float h1 = ninf, h2 = ninf;
        auto fs = [&](float x) {
            h2 = fmaxf(h2, fminf(h1, x));
            h1 = fmax_nan(h1, x);
        };
        if constexpr (ES == 2) {
            uint32_t a1[4] = {kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair};
            uint32_t a2[4] = {kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair, kBf16NegInfPair};
            auto fv = [&](const uint4& u) {
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    a2[q] = bf16x2_max_nan(a2[q], bf16x2_min(a1[q], w[q]));
                    a1[q] = bf16x2_max_nan(a1[q], w[q]);
                }
            };
            if (use_ring) {
                rg.nst = kFirstStages;  // the list region is free until the first read ends
                landed = ring_sweep(rg, row, V * ES, fv);
                rg.nst = kStages;
            }
            else
                sweep_vec<ES>(row, V, fv, fs);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                m1[2 * q] = bf16_lo(a1[q]);
                m1[2 * q + 1] = bf16_hi(a1[q]);
                m2[2 * q] = bf16_lo(a2[q]);
                m2[2 * q + 1] = bf16_hi(a2[q]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < G; ++q) m1[q] = m2[q] = ninf;
            auto fv = [&](const uint4& u) {
                const float x[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                    __uint_as_float(u.w)};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    m2[q] = fmaxf(m2[q], fminf(m1[q], x[q]));
                    m1[q] = fmax_nan(m1[q], x[q]);
                }
            };
            if (use_ring) {
                rg.nst = kFirstStages;  // the list region is free until the first read ends
                landed = ring_sweep(rg, row, V * ES, fv);
                rg.nst = kStages;
            }
            else
                sweep_vec<ES>(row, V, fv, fs);
        }
        m2[0] = fmaxf(fmaxf(m2[0], h2), fminf(m1[0], h1));
        m1[0] = fmax_nan(m1[0], h1);
        float mx = m1[0];
#pragma unroll
        for (int q = 1; q < G; ++q) mx = fmax_nan(mx, m1[q]);
        if (!landed) {
            // A bulk copy did not arrive in time: this row and the CTA's
            // remaining rows report a timeout.
            fail_rows(a, r);
            return;
        }
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
            // The group maxima are distinct elements (an empty group's -inf
            // only lowers the bound), so at least k elements have keys >= the
            // k-th largest of them: to 16 bits it bounds the k-th largest
            // logit from below. A group whose second value is below the
            // bound has at most one element above it, its maximum; a thread
            // with a group that has two or more reads its share again.
            if (t == 0) s.list_n = 0;
            uint32_t lk;
            if (k <= static_cast<uint64_t>(kSortK) && T == 256) {
                // For small k the thread maxima (distinct elements as well)
                // give a bound almost as tight: the CTA sorts them, one per
                // thread (a bitonic network: shuffles within a warp, shared
                // memory across warps), and takes the k-th.
                uint32_t tm = fkey(m1[0]);
#pragma unroll
                for (int q = 1; q < G; ++q) tm = max(tm, fkey(m1[q]));
#pragma unroll
                for (int size = 2; size <= 256; size <<= 1) {
#pragma unroll
                    for (int stride = size >> 1; stride > 0; stride >>= 1) {
                        uint32_t o;
                        if (stride < 32) {
                            o = __shfl_xor_sync(0xFFFFFFFFu, tm, stride);
                        } else {
                            cand[t] = tm;
                            __syncthreads();
                            o = cand[t ^ stride];
                            __syncthreads();
                        }
                        const bool lower = (t & stride) == 0, desc = (t & size) == 0;
                        tm = (lower == desc) ? max(tm, o) : min(tm, o);
                    }
                }
                if (t == static_cast<int>(k) - 1) s.lo = static_cast<int>(tm);
                __syncthreads();
                lk = static_cast<uint32_t>(s.lo);
            } else {
#pragma unroll
                for (int q = 0; q < G; ++q) cand[G * t + q] = fkey(m1[q]);
                __syncthreads();
                lk = (list_select_kth(cand, G * T, k, 2, hc, s) >> 16) << 16;
            }
            bool complete = true;
#pragma unroll
            for (int q = 0; q < G; ++q) complete = complete && fkey(m2[q]) < lk;
            int* inc = reinterpret_cast<int*>(cand);  // the candidates are no longer needed
            if (t == 0) s.inc_n = 0;
            if (__syncthreads_count(!complete) <= kMaxShares) {
                if (complete) {
#pragma unroll
                    for (int q = 0; q < G; ++q) {
                        const uint32_t key = fkey(m1[q]);
                        if (key >= lk) append(key, list, &s.list_n);
                    }
                } else {
                    const int at = atomicAdd(&s.inc_n, 1);
                    if (SV_IN_RANGE(at, kMaxShares)) inc[at] = t;
                    else s.check = kFlagIndex;
                }
                __syncthreads();
                // Many rows need no share read again (about half at k = 50).
                const int ninc = s.inc_n;
                if (ninc > 0) reread_shares<ES>(row, V, inc, ninc, lk, list, &s.list_n);
            } else {
                // Many groups hold two or more elements above the bound (k in the
                // hundreds): one more read of the whole row, a packed compare
                // per 16-byte vector.
                const uint32_t p16 = lk >> 16;
                const bool open = lk <= 0x007FFFFFu;  // the bound is -inf or lower
                const float bound = open ? ninf : key_value(lk);
                const uint32_t b16 = open ? 0xFF80u : bf16_bits_of_key16(p16);
                const uint32_t b2 = b16 | (b16 << 16);
                auto fv = [&](const uint4& u) {
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
                };
                if (use_ring) {
                    __syncthreads();  // the select is done with the bins region
                    if (!ring_sweep(rg, row, V * ES, fv)) {
                        fail_rows(a, r);
                        return;
                    }
                } else {
                    sweep_vec<ES>(row, V, fv, [&](float x) {
                        if (x >= bound) append(fkey(x), list, &s.list_n);
                    });
                }
            }
            __syncthreads();
            const int n = s.list_n;
            if (n <= kSmallList) {
                // One warp selects; the others wait at the barrier below.
                if (t < 32) {
                    uint32_t tw;
                    uint64_t kw;
                    small_select(list, n, tk, k, tp, a.top_p, c, mref, &tw, &kw);
                    if (t == 0) {
                        s.above = kw;
                        s.e = static_cast<int>(tw);
                    }
                }
                __syncthreads();
                tau = static_cast<uint32_t>(s.e);
                kept = s.above;
                done = true;
            } else if (n <= kMidList) {
                mid_select(list, n, k, tp, a.top_p, c, mref, hm, s, &tau, &kept);
                done = true;
            } else if (n <= kListCap) {
                const ListSrc L{list, n};
                tau = list_select_kth(list, n, k, 4, hc, s);
                kept = mass_ge(L, tau, c, mref, s);
                if (tp) {
                    const uint64_t target = static_cast<uint64_t>(
                        ceil(static_cast<double>(a.top_p) * static_cast<double>(kept)));
                    tau = list_select_mass(list, n, 0, target, c, mref, hm, s, &kept);
                }
                done = true;
            }
        } else if (tp && !tk) {
            const int got = topp_bins<ES>(row, V, c, mref, a.top_p, sc, bins, list, s, rg, use_ring,
                                          &tau, &kept);
            rg.buf = smem;  // the ring's usual place
            rg.tile = kTileBytes;
            if (got < 0) {
                fail_rows(a, r);
                return;
            }
            done = got > 0;
        }
        if (!done) row_select<ES>(row, V, tk, k, tp, a.top_p, c, mref, hc, hm, s, &tau, &kept);
        if (t == 0) {
            const float thr = tau == 0u ? ninf : key_value(tau);
            const float l = log2f(__ull2float_rn(kept)) - 40.0f;
            a.rows[r] = FiltRow{mref, l, thr, s.check != 0 ? s.check : (kept > 0 ? 0 : kFlagNonFinite)};
        }
    }
}

}  // namespace

cudaError_t launch_filter(const FilterArgs& a, int grid, int sms, cudaStream_t s)
{
    const bool tk = a.top_k > 0 && a.top_k < a.g.V;
    if (a.g.es == 2 && (!tk || a.top_k > kSortK)) return launch_hist(a, sms, s);
    auto* k = a.g.es == 2 ? filter_kernel<2> : filter_kernel<4>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kFilterSmem));
    if (e != cudaSuccess) return e;
    // The first kernel of a call: launched without programmatic dependent
    // launch, so the caller's earlier work on the stream (the logits) is
    // complete and visible before the first read.
    return launch_dependent(false, k, dim3(static_cast<unsigned>(grid)), dim3(kFilterThreads),
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
