// hist.cu -- top-k / top-p thresholds of bfloat16 rows from an exact count of
// every value in the row, for the cuts the group-maxima kernel (filter.cu)
// does not take: top-p alone, and top-k above 64 (with or without top-p).
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
// A bfloat16 logit is one of 2^16 values, so the count of every value orders
// the whole row: the k-th largest logit, and the mass of every upper set, and
// with it the top-p threshold, follow from the counts alone. One read of the
// row (from HBM, each element once) builds them in shared memory: 2^15 words,
// word g holding the count of +g in its low half and of -g in its high half
// (g the 15 magnitude bits), two shared-memory reductions per pair of
// elements, with a packed maximum for the row maximum and the NaN / +inf
// check. A sweep over the table then gives each thread's 32 magnitudes their
// counts and masses (one exponential per value present, not per element), a
// block-wide scan in value order finds the 32 magnitudes that hold each
// crossing, and one warp walks them to the exact threshold.
//
// A 16-bit count wraps only when 2^16 elements share one value; each wrap
// takes 2^16 - 1 (low half) or 2^16 (high half) from the sum of all counts,
// so the sum equals V exactly when nothing wrapped. A row where it does not
// (a large masked vocabulary, say) is counted again with one 32-bit count per
// magnitude, one sign per read, read from L2.
//
// Masses are integers, so every sum -- and every decision -- is the same on
// every run: a value's mass is 2^(x c - m) 2^40 rounded (m the ceiling of the
// row maximum times c), times its count. The rounding (below 2^-41 of the
// largest mass) and the SFU exponential (a few ulp per value) move a top-p
// boundary by well under 1e-5 of the mass.
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_stages.h"

namespace sv {
namespace {

constexpr int kHT = 1024;                    // threads (32 warps)
constexpr int kHW = kHT / 32;
constexpr int kMags = 32768;                 // table words: one per bfloat16 magnitude
constexpr int kWPT = kMags / kHT;            // words per thread in the table sweeps
static_assert(kWPT == 32, "the crossing walk takes one word per lane");
constexpr int kHU = 8;                       // 16-byte loads in flight per thread
// Dynamic shared memory: the table (128 KB), then the sums of every
// segment of 32 magnitudes (counts and masses of each sign, 24 KB).
constexpr int kSegs = kMags / 32;
constexpr int kHSmem = kMags * 4 + kSegs * (4 + 8 + 4 + 8);
constexpr float kFixH = 1099511627776.0f;    // 2^40

// What the table holds: both signs in 16-bit halves, or one 32-bit count per
// magnitude for the positive values (with -0 as +0) or the negative ones.
enum { kPacked = 0, kPos32 = 1, kNeg32 = 2 };

struct HScratch {
    float wmax[kHW];
    uint32_t wcp[kHW], wcn[kHW];   // per-warp totals, then what lies before each warp
    uint64_t wmp[kHW], wmn[kHW];
    uint32_t tot_pc, tot_nc;       // all positive / negative counts and masses
    uint64_t tot_pm, tot_nm;
    int seg;              // the crossing's 32 magnitudes: thread index, + kHT if negative
    uint32_t seg_c;       // count before them (in value order)
    uint64_t seg_m;       // mass before them
    float tau;            // the threshold found by the walk
    uint64_t through;     // mass of the upper set {x >= tau}
    int fail;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void red_add(uint32_t addr, uint32_t v)
{
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v));
}

// A 16-byte load that allocates no L1 line (each row is read once here).
__device__ __forceinline__ uint4 ldg_stream(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Fixed-point mass of one token: 2^(x c - m) 2^40, rounded.
__device__ __forceinline__ uint64_t mass_fix(float x, float c, float m)
{
    return __float2ull_rn(ex2(fmaf(x, c, -m)) * kFixH);
}

// ceil(top_p * mass) for top_p in (0, 1), exactly, in integer arithmetic:
// top_p = f 2^-e with f its 24-bit significand, so the product is f mass / 2^e.
__device__ __forceinline__ uint64_t ceil_frac(float top_p, uint64_t mass)
{
    const uint32_t bits = __float_as_uint(top_p);
    const int ex = static_cast<int>((bits >> 23) & 0xFFu);
    const uint64_t f = ex ? ((bits & 0x7FFFFFu) | 0x800000u) : (bits & 0x7FFFFFu);
    const int e = 150 - (ex ? ex : 1);  // e >= 24 for top_p < 1
    const uint64_t lo = f * mass, hi = __umul64hi(f, mass);
    if (e >= 128) return (lo | hi) ? 1u : 0u;
    uint64_t q;
    bool rem;
    if (e >= 64) {
        q = hi >> (e - 64);
        rem = lo != 0 || (e > 64 && (hi & ((uint64_t(1) << (e - 64)) - 1)) != 0);
    } else {
        q = (lo >> e) | (hi << (64 - e));
        rem = (lo & ((uint64_t(1) << e) - 1)) != 0;
    }
    return q + (rem ? 1u : 0u);
}

// Adds the two elements of a 32-bit word to the packed table: the low
// element at word (w & 0x7FFF), the high one at word ((w >> 16) & 0x7FFF);
// +1 for a positive value, +2^16 for a negative one (prmt replicates the sign
// bit of byte 1 or byte 3 into 0xFFFF, which plus one is 2^16).
__device__ __forceinline__ void count_pair(uint32_t base, uint32_t w)
{
    red_add(base + ((w & 0x7FFFu) << 2), prmt(w, 0u, 0x4499u) + 1u);
    red_add(base + ((w >> 14) & 0x1FFFCu), prmt(w, 0u, 0x44BBu) + 1u);
}

// One element given by its 16 bits, in table mode MODE.
template <int MODE>
__device__ __forceinline__ void count_one(uint32_t base, uint32_t h)
{
    const uint32_t addr = base + ((h & 0x7FFFu) << 2);
    const bool neg = (h & 0x8000u) != 0u && h != 0x8000u;  // -0 counts as +0
    if (MODE == kPacked) red_add(addr, (h & 0x8000u) ? 0x10000u : 1u);
    else if (MODE == kPos32) { if (!neg) red_add(addr, 1u); }
    else { if (neg) red_add(addr, 1u); }
}

template <int MODE>
__device__ __forceinline__ void count_word(uint32_t base, uint32_t w)
{
    if (MODE == kPacked) {
        count_pair(base, w);
    } else {
        count_one<MODE>(base, w & 0xFFFFu);
        count_one<MODE>(base, w >> 16);
    }
}

__device__ __forceinline__ void zero_table(uint32_t* tab)
{
    uint4* t4 = reinterpret_cast<uint4*>(tab);
    for (int i = threadIdx.x; i < kMags / 4; i += kHT) t4[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Counts one row (V bfloat16 values, 2-byte aligned) into the zeroed table.
// In packed mode also returns this thread's NaN-propagating maximum.
template <int MODE>
__device__ void count_row(const uint8_t* row, int64_t V, uint32_t base, float* tmax)
{
    const int t = threadIdx.x;
    const uint16_t* r16 = reinterpret_cast<const uint16_t*>(row);
    const uintptr_t rp = reinterpret_cast<uintptr_t>(row);
    int64_t head = static_cast<int64_t>(((16u - static_cast<uint32_t>(rp & 15u)) & 15u) >> 1);
    if (head > V) head = V;
    const int64_t nvec = (V - head) >> 3;
    const int64_t tail = head + (nvec << 3);
    const uint4* vp = reinterpret_cast<const uint4*>(row + head * 2);
    uint32_t pm = kBf16NegInfPair;
    for (int64_t v0 = 0; v0 < nvec; v0 += static_cast<int64_t>(kHU) * kHT) {
        uint4 u[kHU];
#pragma unroll
        for (int q = 0; q < kHU; ++q) {
            const int64_t v = v0 + q * kHT + t;
            u[q] = v < nvec ? ldg_stream(vp + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kHU; ++q) {
            if (v0 + q * kHT + t < nvec) {
                count_word<MODE>(base, u[q].x);
                count_word<MODE>(base, u[q].y);
                count_word<MODE>(base, u[q].z);
                count_word<MODE>(base, u[q].w);
                if (MODE == kPacked)
                    pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(u[q].x, u[q].y),
                                                           bf16x2_max_nan(u[q].z, u[q].w)));
            }
        }
    }
    float m = fmax_nan(bf16_lo(pm), bf16_hi(pm));
    for (int64_t i = t; i < head; i += kHT) {
        const uint32_t h = r16[i];
        count_one<MODE>(base, h);
        m = fmax_nan(m, __uint_as_float(h << 16));
    }
    for (int64_t i = tail + t; i < V; i += kHT) {
        const uint32_t h = r16[i];
        count_one<MODE>(base, h);
        m = fmax_nan(m, __uint_as_float(h << 16));
    }
    if (tmax != nullptr) *tmax = m;
}

// Counts of magnitude g from its table word: (positive, negative), with -0
// merged into +0.
template <int MODE>
__device__ __forceinline__ void split_word(uint32_t w, uint32_t g, uint32_t* np, uint32_t* nn)
{
    if (MODE == kPacked) {
        *np = w & 0xFFFFu;
        *nn = w >> 16;
        if (g == 0u) {
            *np += *nn;
            *nn = 0u;
        }
    } else if (MODE == kPos32) {
        *np = w;
        *nn = 0u;
    } else {
        *np = 0u;
        *nn = w;
    }
}

// Counts and masses of the positive and of the negative values of every
// segment of 32 magnitudes [32 j, 32 j + 32), into the segment arrays. Warp w
// takes the segments j = w (mod 32), one magnitude per lane, so that the few
// dense segments near the bulk of a row spread over all warps; an empty
// segment costs one vote, a non-empty one a warp reduction.
struct SegArrays {
    uint32_t* cp;
    uint64_t* mp;
    uint32_t* cn;
    uint64_t* mn;
};

template <int MODE>
__device__ void segment_sums(const uint32_t* tab, float c, float mref, const SegArrays& A)
{
    const uint32_t lane = threadIdx.x & 31u, w = threadIdx.x >> 5;
    for (uint32_t j = w; j < static_cast<uint32_t>(kSegs); j += kHW) {
        const uint32_t g = 32u * j + lane;
        const uint32_t word = tab[g];
        if (!__any_sync(0xFFFFFFFFu, word != 0u)) {
            if (lane == 0) {
                A.cp[j] = 0u;
                A.mp[j] = 0u;
                A.cn[j] = 0u;
                A.mn[j] = 0u;
            }
            continue;
        }
        uint32_t np, nn;
        split_word<MODE>(word, g, &np, &nn);
        const float v = __uint_as_float(g << 16);
        uint64_t mp = np ? static_cast<uint64_t>(np) * mass_fix(v, c, mref) : 0u;
        uint64_t mn = nn ? static_cast<uint64_t>(nn) * mass_fix(-v, c, mref) : 0u;
        uint64_t cc = (static_cast<uint64_t>(np) << 32) | nn;  // counts below 2^21 each
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            cc += __shfl_xor_sync(0xFFFFFFFFu, cc, off);
            mp += __shfl_xor_sync(0xFFFFFFFFu, mp, off);
            mn += __shfl_xor_sync(0xFFFFFFFFu, mn, off);
        }
        if (lane == 0) {
            A.cp[j] = static_cast<uint32_t>(cc >> 32);
            A.mp[j] = mp;
            A.cn[j] = static_cast<uint32_t>(cc);
            A.mn[j] = mn;
        }
    }
}

// Block-wide positions of every thread's two segments in value order: the
// positive segments from the largest magnitudes down (thread kHT - 1 first),
// then the negative ones from the smallest magnitude up (thread 0 first).
// Returns the count and mass before each segment and the grand totals.
struct SegPos {
    uint32_t bcp, bcn;    // count before this thread's positive / negative segment
    uint64_t bmp, bmn;    // mass before them
    uint32_t tot_c;
    uint64_t tot_m;
};

__device__ SegPos segment_positions(uint32_t cp, uint64_t mp, uint32_t cn, uint64_t mn,
                                    HScratch& s)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    // Within the warp: positive, suffix sums over the lanes; negative, prefix sums.
    uint32_t sc = cp, pc = cn;
    uint64_t sm = mp, pmv = mn;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t oc = __shfl_down_sync(0xFFFFFFFFu, sc, off);
        const uint64_t om = __shfl_down_sync(0xFFFFFFFFu, sm, off);
        const uint32_t qc = __shfl_up_sync(0xFFFFFFFFu, pc, off);
        const uint64_t qm = __shfl_up_sync(0xFFFFFFFFu, pmv, off);
        if (lane + off < 32) {
            sc += oc;
            sm += om;
        }
        if (lane >= off) {
            pc += qc;
            pmv += qm;
        }
    }
    __syncthreads();  // the scratch of the previous use has been read
    if (lane == 0) {
        s.wcp[w] = sc;
        s.wmp[w] = sm;
    }
    if (lane == 31) {
        s.wcn[w] = pc;
        s.wmn[w] = pmv;
    }
    __syncthreads();
    // Warp 0: what lies before each warp, and the totals.
    if (w == 0) {
        const uint32_t c1 = s.wcp[lane], c2 = s.wcn[lane];
        const uint64_t m1 = s.wmp[lane], m2 = s.wmn[lane];
        uint32_t a1 = c1, a2 = c2;
        uint64_t b1 = m1, b2 = m2;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t oc = __shfl_down_sync(0xFFFFFFFFu, a1, off);
            const uint64_t om = __shfl_down_sync(0xFFFFFFFFu, b1, off);
            const uint32_t qc = __shfl_up_sync(0xFFFFFFFFu, a2, off);
            const uint64_t qm = __shfl_up_sync(0xFFFFFFFFu, b2, off);
            if (lane + off < 32) {
                a1 += oc;
                b1 += om;
            }
            if (lane >= off) {
                a2 += qc;
                b2 += qm;
            }
        }
        __syncwarp();
        s.wcp[lane] = a1 - c1;  // positive: the warps above this one
        s.wmp[lane] = b1 - m1;
        s.wcn[lane] = a2 - c2;  // negative: the warps below this one
        s.wmn[lane] = b2 - m2;
        if (lane == 0) {
            s.tot_pc = a1;
            s.tot_pm = b1;
        }
        if (lane == 31) {
            s.tot_nc = a2;
            s.tot_nm = b2;
        }
    }
    __syncthreads();
    SegPos r;
    r.bcp = s.wcp[w] + (sc - cp);
    r.bmp = s.wmp[w] + (sm - mp);
    r.bcn = s.tot_pc + s.wcn[w] + (pc - cn);
    r.bmn = s.tot_pm + s.wmn[w] + (pmv - mn);
    r.tot_c = s.tot_pc + s.tot_nc;
    r.tot_m = s.tot_pm + s.tot_nm;
    return r;
}

// The segment (of 32 magnitudes, one sign) where the running count (BY_MASS
// false) or mass (true) in value order first reaches `need`: the thread that
// owns it records it. Exactly one segment qualifies when 0 < need <= total.
template <bool BY_MASS>
__device__ __forceinline__ void claim_segment(const SegPos& p, uint32_t cp, uint64_t mp, uint32_t cn,
                                              uint64_t mn, uint64_t need, HScratch& s)
{
    if (BY_MASS) {
        if (p.bmp < need && need <= p.bmp + mp && mp > 0) {
            s.seg = threadIdx.x;
            s.seg_c = p.bcp;
            s.seg_m = p.bmp;
        }
        if (p.bmn < need && need <= p.bmn + mn && mn > 0) {
            s.seg = threadIdx.x + kHT;
            s.seg_c = p.bcn;
            s.seg_m = p.bmn;
        }
    } else {
        if (p.bcp < need && need <= p.bcp + cp) {
            s.seg = threadIdx.x;
            s.seg_c = p.bcp;
            s.seg_m = p.bmp;
        }
        if (p.bcn < need && need <= p.bcn + cn) {
            s.seg = threadIdx.x + kHT;
            s.seg_c = p.bcn;
            s.seg_m = p.bmn;
        }
    }
}

// Warp 0: walks the claimed segment, one magnitude per lane in value order,
// to the first value where the running count or mass reaches `need`; records
// that value and the mass of its upper set. The table must hold the
// segment's sign (packed, or the matching 32-bit mode).
template <int MODE, bool BY_MASS>
__device__ void walk_segment(const uint32_t* tab, float c, float mref, uint64_t need, HScratch& s)
{
    const uint32_t lane = threadIdx.x & 31u;
    const int seg = s.seg;
    const bool pos = seg < kHT;
    const uint32_t owner = static_cast<uint32_t>(pos ? seg : seg - kHT);
    // Positive values descend with the magnitude, negative ones ascend.
    const uint32_t g = owner * kWPT + (pos ? 31u - lane : lane);
    uint32_t np, nn;
    split_word<MODE>(tab[g], g, &np, &nn);
    const uint32_t n = pos ? np : nn;
    const float v = pos ? __uint_as_float(g << 16) : -__uint_as_float(g << 16);
    const uint64_t m = n ? static_cast<uint64_t>(n) * mass_fix(v, c, mref) : 0u;
    uint64_t cc = n, cm = m;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t oc = __shfl_up_sync(0xFFFFFFFFu, cc, off);
        const uint64_t om = __shfl_up_sync(0xFFFFFFFFu, cm, off);
        if (lane >= static_cast<uint32_t>(off)) {
            cc += oc;
            cm += om;
        }
    }
    const bool hit = BY_MASS ? (s.seg_m + cm >= need) : (s.seg_c + cc >= need);
    const unsigned b = __ballot_sync(0xFFFFFFFFu, hit);
    if (b != 0u && lane == static_cast<uint32_t>(__ffs(b) - 1)) {
        s.tau = v == 0.0f ? 0.0f : v;
        s.through = s.seg_m + cm;
    }
}

__device__ __forceinline__ float block_max(float m, HScratch& s)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    __syncthreads();
    if (lane == 0) s.wmax[w] = m;
    __syncthreads();
    float r = s.wmax[0];
    for (int v = 1; v < kHW; ++v) r = fmax_nan(r, s.wmax[v]);
    return r;
}

// Per-row constants of the selection.
struct CutK {
    bool tk, tp;
    uint64_t k;
    float top_p;
    float c;
};

// The thresholds of one counted row. Every thread calls it, with its segment
// sums; the table holds the packed counts (MODE kPacked) or one sign's 32-bit
// counts (*mode_now), and is counted again when the other sign is needed.
// False if no segment holds a crossing (impossible with exact integer sums;
// the row is then reported as failed rather than read out of range).
template <int MODE>
__device__ bool select_row(const uint8_t* row, int64_t V, uint32_t* tab, uint32_t base,
                           const CutK& P, float mref, const SegPos& pos, uint32_t cp, uint64_t mp,
                           uint32_t cn, uint64_t mn, int* mode_now, HScratch& s, float* tau,
                           uint64_t* kept)
{
    // Makes the table hold the sign of the claimed segment (32-bit modes).
    auto hold_sign = [&]() {
        if (MODE == kPacked) return;
        const int want = s.seg < kHT ? kPos32 : kNeg32;
        if (*mode_now == want) return;
        __syncthreads();
        zero_table(tab);
        __syncthreads();
        if (want == kPos32) count_row<kPos32>(row, V, base, nullptr);
        else count_row<kNeg32>(row, V, base, nullptr);
        __syncthreads();
        *mode_now = want;
    };
    auto walk = [&](bool by_mass, uint64_t need) {
        if (threadIdx.x < 32) {
            const int m = MODE == kPacked ? kPacked : *mode_now;
            if (m == kPacked) {
                if (by_mass) walk_segment<kPacked, true>(tab, P.c, mref, need, s);
                else walk_segment<kPacked, false>(tab, P.c, mref, need, s);
            } else if (m == kPos32) {
                if (by_mass) walk_segment<kPos32, true>(tab, P.c, mref, need, s);
                else walk_segment<kPos32, false>(tab, P.c, mref, need, s);
            } else {
                if (by_mass) walk_segment<kNeg32, true>(tab, P.c, mref, need, s);
                else walk_segment<kNeg32, false>(tab, P.c, mref, need, s);
            }
        }
        __syncthreads();
    };

    float t_val = __uint_as_float(kF32NegInfBits);
    uint64_t mass_k = pos.tot_m;
    if (P.tk) {
        if (threadIdx.x == 0) s.seg = -1;
        __syncthreads();
        claim_segment<false>(pos, cp, mp, cn, mn, P.k, s);
        __syncthreads();
        if (s.seg < 0) return false;
        hold_sign();
        walk(false, P.k);
        t_val = s.tau;
        mass_k = s.through;
    }
    if (P.tp) {
        const uint64_t target = ceil_frac(P.top_p, mass_k);
        __syncthreads();  // every thread has read s.tau / s.through
        if (threadIdx.x == 0) s.seg = -1;
        __syncthreads();
        claim_segment<true>(pos, cp, mp, cn, mn, target, s);
        __syncthreads();
        if (s.seg < 0) return false;
        hold_sign();
        walk(true, target);
        t_val = s.tau;
        *kept = s.through;
    } else {
        *kept = mass_k;
    }
    *tau = t_val;
    return true;
}

__device__ void fail_rows(const FilterArgs& a, int flags)
{
    if (threadIdx.x != 0) return;
    for (int64_t r = blockIdx.x; r < a.g.rows; r += gridDim.x) a.rows[r] = FiltRow{0.f, 0.f, 0.f, flags};
}

__global__ void __launch_bounds__(kHT, 1) hist_kernel(const __grid_constant__ FilterArgs a)
{
    extern __shared__ __align__(16) uint32_t tab[];
    __shared__ HScratch s;
    const SegArrays A{tab + kMags, reinterpret_cast<uint64_t*>(tab + kMags + kSegs),
                      tab + kMags + 3 * kSegs, reinterpret_cast<uint64_t*>(tab + kMags + 4 * kSegs)};
    const int t = threadIdx.x;
    const int64_t V = a.g.V;
    const uint32_t base = smem_addr(tab);
    CutK P;
    P.tk = a.top_k > 0 && a.top_k < V;
    P.tp = a.top_p < 1.0f;
    P.k = P.tk ? static_cast<uint64_t>(a.top_k) : 0u;
    P.top_p = a.top_p;
    P.c = a.c;
    pdl_trigger();  // the scan may launch; it waits for this grid before reading
    if (a.gate != nullptr) {
        // Test hook: hold every read until *gate != 0, bounded like every
        // other wait. Nothing sets it in the tests that use it: the CTA then
        // marks its rows as timed out and returns.
        if (t == 0) {
            s.fail = 0;
            const volatile int32_t* gate = a.gate;
            const long long t0 = clock64();
            while (*gate == 0) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    s.fail = 1;
                    break;
                }
                __nanosleep(1000);
            }
        }
        __syncthreads();
        if (s.fail != 0) {
            fail_rows(a, kFlagTimeout);
            return;
        }
    }

    for (int64_t r = blockIdx.x; r < a.g.rows; r += gridDim.x) {
        const uint8_t* row = r < a.g.rows_t ? a.target + r * V * 2 : a.draft + (r - a.g.rows_t) * V * 2;
        __syncthreads();  // the previous row is done with the table
        zero_table(tab);
        __syncthreads();
        float tm;
        count_row<kPacked>(row, V, base, &tm);
        const float mx = block_max(tm, s);  // its barriers also order the counts before the sweep
        if (!(mx > __uint_as_float(kF32NegInfBits)) || !(mx < __uint_as_float(0x7F800000u))) {
            // NaN or +inf in the row, or no finite logit.
            if (t == 0) a.rows[r] = FiltRow{0.f, 0.f, 0.f, kFlagNonFinite};
            continue;
        }
        const float mref = ceilf(mx * P.c);
        // This thread's segment (magnitudes [32 t, 32 t + 32)): its sums.
        auto own_sums = [&](uint32_t* cp, uint64_t* mp, uint32_t* cn, uint64_t* mn) {
            __syncthreads();  // the segment arrays are written
            *cp = A.cp[t];
            *mp = A.mp[t];
            *cn = A.cn[t];
            *mn = A.mn[t];
        };
        uint32_t cp, cn;
        uint64_t mp, mn;
        segment_sums<kPacked>(tab, P.c, mref, A);
        own_sums(&cp, &mp, &cn, &mn);
        SegPos pos = segment_positions(cp, mp, cn, mn, s);
        float tau = 0.f;
        uint64_t kept = 0;
        bool ok;
        if (pos.tot_c == static_cast<uint64_t>(V)) {
            int mode_now = kPacked;
            ok = select_row<kPacked>(row, V, tab, base, P, mref, pos, cp, mp, cn, mn, &mode_now, s,
                                     &tau, &kept);
        } else {
            // A 16-bit count wrapped (the counts fall short of V): count
            // again, one sign per read, 32 bits per magnitude.
            zero_table(tab);
            __syncthreads();
            count_row<kPos32>(row, V, base, nullptr);
            __syncthreads();
            segment_sums<kPos32>(tab, P.c, mref, A);
            uint32_t c2, c3;
            uint64_t m2, m3;
            own_sums(&cp, &mp, &c2, &m2);
            zero_table(tab);
            __syncthreads();
            count_row<kNeg32>(row, V, base, nullptr);
            __syncthreads();
            segment_sums<kNeg32>(tab, P.c, mref, A);
            own_sums(&c2, &m2, &c3, &m3);
            cn = c3;
            mn = m3;
            pos = segment_positions(cp, mp, cn, mn, s);
            int mode_now = kNeg32;
            ok = select_row<kNeg32>(row, V, tab, base, P, mref, pos, cp, mp, cn, mn, &mode_now, s,
                                    &tau, &kept);
        }
        if (t == 0) {
            const float l = log2f(__ull2float_rn(kept)) - 40.0f;
            a.rows[r] = ok && kept > 0 ? FiltRow{mref, l, tau, 0} : FiltRow{0.f, 0.f, 0.f, kFlagNonFinite};
        }
    }
}

}  // namespace

cudaError_t launch_hist(const FilterArgs& a, int sms, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = a.g.rows < sms ? a.g.rows : sms;
    if (grid <= 0) return cudaSuccess;
    // The first kernel of a call: launched without programmatic dependent
    // launch, so the caller's earlier work on the stream (the logits) is
    // complete and visible before the first read.
    return launch_dependent(false, hist_kernel, dim3(static_cast<unsigned>(grid)), dim3(kHT),
                            static_cast<size_t>(kHSmem), s, a);
}

}  // namespace sv
