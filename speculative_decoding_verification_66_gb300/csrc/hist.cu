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
// row (from HBM, each element once) counts its values in shared memory, two
// shared-memory reductions per pair of elements plus a packed maximum (the row
// maximum, and the NaN / +inf check). The table is a window of 2^14 words over
// the magnitudes of 128 binades, 2^-64 <= |x| < 2^64, word g holding the count
// of +g in its low half and of -g in its high half; two more words count the
// magnitudes below the window (zeros, mostly) and above it (-inf, mostly).
// Two CTAs share an SM, so that one's selection runs while the other counts
// (the counting is bound by the SM's shared-memory atomics).
//
// The selection: the 2^10 segments of 32 magnitudes of each sign get their
// counts and masses (one exponential per value present, not per element); a
// block-wide scan in value order finds the segment that holds each crossing,
// and one warp walks it to the exact threshold.
//
// Three things send a row to a slower exact path that counts it again, with
// one 32-bit count per magnitude, in four reads (one sign and half of the
// magnitudes each, from L2): a 16-bit count that wrapped (2^16 elements share
// a value; each wrap takes 2^16 - 1 or 2^16 from the sum of all counts, so the
// sum equals V exactly when nothing wrapped), a crossing among the values
// outside the window, or a row maximum of 2^64 or more.
//
// Masses are integers, so every sum -- and every decision -- is the same on
// every run: the mass of a value's n tokens is n 2^(x c - m) on a grid of
// 2^-40 (m the ceiling of the row maximum times c), the bits below the grid
// dropped; a value below the window has the mass of 0, one above it (below
// -2^64) none. The truncation (below 2^-40 of the largest mass, per value)
// and the SFU exponential (a few ulp per value) move a top-p boundary by well
// under 1e-5 of the mass.
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_stages.h"

namespace sv {
namespace {

constexpr int kHT = 512;                     // threads (16 warps); two CTAs per SM
constexpr int kHW = kHT / 32;
constexpr uint32_t kG0 = 63u * 128u;         // first magnitude of the window (2^-64)
constexpr int kWin = 16384;                  // magnitudes in the window
constexpr int kSegs = 1024;                  // segments of 32 magnitudes, per sign
constexpr int kHU = 8;                       // 16-byte loads in flight per thread

// Dynamic shared memory: 16 bytes whose last word counts the magnitudes below
// the window, the window (64 KB), 16 bytes whose first word counts those
// above it, then the sums of every segment (counts and masses of each sign).
constexpr int kTabBytes = 16 + kWin * 4 + 16;
constexpr int kHSmem = kTabBytes + kSegs * (4 + 8 + 4 + 8);

// What the table holds: the window, both signs in 16-bit halves; or 32-bit
// counts of one sign and half of the magnitudes (kQ0 + 2 sign + half), with
// -0 counted as +0.
enum { kPacked = -1, kQ0 = 0, kQ1 = 1, kQ2 = 2, kQ3 = 3 };

struct HScratch {
    float wmax[kHW];
    uint32_t sum_c[kHW];           // block_sum2's per-warp sums (its own slots: the
    uint64_t sum_m[kHW];           // scan that follows writes wcp / wmp at once)
    uint32_t wcp[kHW], wcn[kHW];   // per-warp totals, then what lies before each warp
    uint64_t wmp[kHW], wmn[kHW];
    uint32_t tot_pc, tot_nc;       // all positive / negative counts and masses
    uint64_t tot_pm, tot_nm;
    int seg[2];           // the crossing's segment (top-k, top-p): index, + kSegs if negative; -1 none
    uint32_t seg_c[2];    // count before it (in value order)
    uint64_t seg_m[2];    // mass before it
    float tau;            // the threshold found by the walk or the scan
    uint64_t through;     // mass of the upper set {x >= tau}
    int found;            // the scan: 0 not yet, 1 found, 2 in an outer word
    int fail;
    int check;            // kFlagIndex when a device-side index check failed on this row
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

// Fixed-point mass of n tokens of logit x: n 2^(x c - m) in units of 2^-40,
// from the bits of the float y = 2^(x c - m) <= 1 (x at most the row maximum):
// its 24-bit significand times n, shifted to the 2^-40 grid (the part below
// it dropped). Integer work only, after the exponential.
__device__ __forceinline__ uint64_t mass_n(uint32_t n, float x, float c, float m)
{
    const uint32_t b = __float_as_uint(ex2(fmaf(x, c, -m)));
    const int e = static_cast<int>(b >> 23);  // biased; 0 for a flushed subnormal or 0
    const uint64_t f = static_cast<uint64_t>(n) * ((b & 0x7FFFFFu) | (e ? 0x800000u : 0u));
    // y = f 2^(e - 150), so y 2^40 = f 2^(e - 110).
    const int sh = e - 110;
    return sh >= 0 ? f << sh : (sh > -64 ? f >> -sh : 0u);
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

// Shared address of the window word of magnitude g; magnitudes below the
// window go to the word before it, those above to the word after it.
__device__ __forceinline__ uint32_t win_addr(uint32_t win, uint32_t g)
{
    int i = static_cast<int>(g) - static_cast<int>(kG0);
    i = max(-1, min(i, kWin));
    return win + static_cast<uint32_t>(i * 4);
}

__device__ __forceinline__ uint32_t umin16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Adds the two elements of a 32-bit word to the packed window: +1 for a
// positive value, +2^16 for a negative one (prmt replicates the sign bit of
// byte 1 or byte 3 into 0xFFFF, which plus one is 2^16). Both word indices
// come out of one packed computation: each magnitude g, offset by 2^15 - kG0
// (no half can carry), clamped to [2^15 - 1, 2^15 + kWin], is 2^15 plus its
// window index as win_addr clamps it; win_b is the window's address minus
// 4 2^15.
__device__ __forceinline__ void count_pair(uint32_t win_b, uint32_t w)
{
    constexpr uint32_t kBias = (0x8000u - kG0) * 0x10001u;
    constexpr uint32_t kLo = 0x7FFFu * 0x10001u, kHi = (0x8000u + kWin) * 0x10001u;
    const uint32_t i2 = umin16x2(umax16x2((w & 0x7FFF7FFFu) + kBias, kLo), kHi);
    red_add(win_b + ((i2 & 0xFFFFu) << 2), prmt(w, 0u, 0x4499u) + 1u);
    red_add(win_b + ((i2 >> 16) << 2), prmt(w, 0u, 0x44BBu) + 1u);
}

// One element given by its 16 bits, in table mode MODE.
template <int MODE>
__device__ __forceinline__ void count_one(uint32_t win, uint32_t h)
{
    if (MODE == kPacked) {
        red_add(win_addr(win, h & 0x7FFFu), (h & 0x8000u) ? 0x10000u : 1u);
    } else {
        const bool neg = (h & 0x8000u) != 0u && h != 0x8000u;  // -0 counts as +0
        const uint32_t i = (h & 0x7FFFu) - (MODE & 1 ? static_cast<uint32_t>(kWin) : 0u);
        if (neg == (MODE >= kQ2) && i < static_cast<uint32_t>(kWin)) red_add(win + i * 4u, 1u);
    }
}

template <int MODE>
__device__ __forceinline__ void count_word(uint32_t win, uint32_t w)
{
    if (MODE == kPacked) {
        count_pair(win - 4u * 0x8000u, w);
    } else {
        count_one<MODE>(win, w & 0xFFFFu);
        count_one<MODE>(win, w >> 16);
    }
}

// Zeroes the window and the two words beside it.
__device__ __forceinline__ void zero_table(uint8_t* tabmem)
{
    uint4* t4 = reinterpret_cast<uint4*>(tabmem);
    for (int i = threadIdx.x; i < kTabBytes / 16; i += kHT) t4[i] = make_uint4(0u, 0u, 0u, 0u);
}

// A row of V bfloat16 values (2-byte aligned) as 16-byte vectors, with the
// elements before the first 16-byte boundary (head) and after the last
// whole vector (tail) apart.
struct RowVecs {
    const uint16_t* r16;
    const uint4* vp;
    int64_t head, nvec, tail, V;
};

__device__ __forceinline__ RowVecs row_vecs(const uint8_t* row, int64_t V)
{
    RowVecs rv;
    rv.r16 = reinterpret_cast<const uint16_t*>(row);
    const uintptr_t rp = reinterpret_cast<uintptr_t>(row);
    rv.head = static_cast<int64_t>(((16u - static_cast<uint32_t>(rp & 15u)) & 15u) >> 1);
    if (rv.head > V) rv.head = V;
    rv.nvec = (V - rv.head) >> 3;
    rv.tail = rv.head + (rv.nvec << 3);
    rv.vp = reinterpret_cast<const uint4*>(row + rv.head * 2);
    rv.V = V;
    return rv;
}

// This thread's vectors v0 + q kHT + t of a batch (zeros past the end).
__device__ __forceinline__ void load_batch(const RowVecs& rv, int64_t v0, uint4 (&u)[kHU])
{
#pragma unroll
    for (int q = 0; q < kHU; ++q) {
        const int64_t v = v0 + q * kHT + threadIdx.x;
        u[q] = v < rv.nvec ? ldg_stream(rv.vp + v) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Counts a row into the zeroed table. With PRE, u already holds the first
// batch (loaded before the table was cleared, so that those loads overlap
// it). In packed mode also returns this thread's NaN-propagating maximum.
template <int MODE, bool PRE>
__device__ __forceinline__ void count_vecs(const RowVecs& rv, uint32_t win, uint4 (&u)[kHU],
                                           float* tmax)
{
    const int t = threadIdx.x;
    uint32_t pm = kBf16NegInfPair;
    for (int64_t v0 = 0; v0 < rv.nvec; v0 += static_cast<int64_t>(kHU) * kHT) {
        if (!PRE || v0 != 0) load_batch(rv, v0, u);
#pragma unroll
        for (int q = 0; q < kHU; ++q) {
            if (v0 + q * kHT + t < rv.nvec) {
                count_word<MODE>(win, u[q].x);
                count_word<MODE>(win, u[q].y);
                count_word<MODE>(win, u[q].z);
                count_word<MODE>(win, u[q].w);
                if (MODE == kPacked)
                    pm = bf16x2_max_nan(pm, bf16x2_max_nan(bf16x2_max_nan(u[q].x, u[q].y),
                                                           bf16x2_max_nan(u[q].z, u[q].w)));
            }
        }
    }
    float m = fmax_nan(bf16_lo(pm), bf16_hi(pm));
    for (int64_t i = t; i < rv.head; i += kHT) {
        const uint32_t h = rv.r16[i];
        count_one<MODE>(win, h);
        m = fmax_nan(m, __uint_as_float(h << 16));
    }
    for (int64_t i = rv.tail + t; i < rv.V; i += kHT) {
        const uint32_t h = rv.r16[i];
        count_one<MODE>(win, h);
        m = fmax_nan(m, __uint_as_float(h << 16));
    }
    if (tmax != nullptr) *tmax = m;
}

// Counts one row (V bfloat16 values, 2-byte aligned) into the zeroed table.
template <int MODE>
__device__ void count_row(const uint8_t* row, int64_t V, uint32_t win)
{
    uint4 u[kHU];
    count_vecs<MODE, false>(row_vecs(row, V), win, u, nullptr);
}

// First magnitude that word 0 of a 32-bit table stands for, in mode MODE.
template <int MODE>
__device__ __forceinline__ uint32_t table_g0()
{
    return MODE & 1 ? static_cast<uint32_t>(kWin) : 0u;
}

// The counts a 32-bit table word gives magnitude g's positive and negative
// value.
template <int MODE>
__device__ __forceinline__ void split_word(uint32_t w, uint32_t* np, uint32_t* nn)
{
    if (MODE < kQ2) {
        *np = w;
        *nn = 0u;
    } else {
        *np = 0u;
        *nn = w;
    }
}

struct SegArrays {
    uint32_t* cp;   // [kSegs] per segment: positive count
    uint64_t* mp;   //                      positive mass
    uint32_t* cn;   //                      negative count
    uint64_t* mn;   //                      negative mass
};

// The sums of a 32-bit table's 512 segments into the segment arrays (global
// segment = table_g0 / 32 + local). Warp w takes blocks of 4 segments (one
// 16-byte load per lane, 8 lanes per segment), blocks w, w + 16, ...; an
// empty block costs one vote, a non-empty one a reduction over 8 lanes.
template <int MODE>
__device__ void segment_sums(const uint32_t* win, float c, float mref, const SegArrays& A)
{
    const uint32_t lane = threadIdx.x & 31u, w = threadIdx.x >> 5;
    const uint32_t g0 = table_g0<MODE>();
    const uint4* w4 = reinterpret_cast<const uint4*>(win);
    for (uint32_t b = w; b < static_cast<uint32_t>(kWin / 128); b += kHW) {
        const uint4 q = w4[32u * b + lane];
        const uint32_t j = g0 / 32u + 4u * b + (lane >> 3);  // this lane's segment
        const bool nz = (q.x | q.y | q.z | q.w) != 0u;
        uint32_t c_p = 0, c_n = 0;
        uint64_t m_p = 0, m_n = 0;
        if (__any_sync(0xFFFFFFFFu, nz)) {
            if (nz) {
                const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t np, nn;
                    split_word<MODE>(ws[k], &np, &nn);
                    const uint32_t g = g0 + 128u * b + 4u * lane + static_cast<uint32_t>(k);
                    const float v = __uint_as_float(g << 16);
                    if (np) {
                        c_p += np;
                        m_p += mass_n(np, v, c, mref);
                    }
                    if (nn) {
                        c_n += nn;
                        m_n += mass_n(nn, -v, c, mref);
                    }
                }
            }
            uint64_t cc = (static_cast<uint64_t>(c_p) << 32) | c_n;  // counts below 2^22 each
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) {
                cc += __shfl_xor_sync(0xFFFFFFFFu, cc, off);
                m_p += __shfl_xor_sync(0xFFFFFFFFu, m_p, off);
                m_n += __shfl_xor_sync(0xFFFFFFFFu, m_n, off);
            }
            c_p = static_cast<uint32_t>(cc >> 32);
            c_n = static_cast<uint32_t>(cc);
        }
        if ((lane & 7u) == 0u) {
            if (MODE < kQ2) {
                A.cp[j] = c_p;
                A.mp[j] = m_p;
            } else {
                A.cn[j] = c_n;
                A.mn[j] = m_n;
            }
        }
    }
}

// A thread's two segments 2t, 2t + 1 of each sign.
struct OwnSegs {
    uint32_t cp[2], cn[2];
    uint64_t mp[2], mn[2];
};

// Block-wide positions of every thread's segments in value order: the
// positive ones from the largest magnitudes down (thread kHT - 1 first), then
// the negative ones from the smallest magnitude up (thread 0 first).
struct SegPos {
    uint32_t bcp, bcn;    // count before this thread's positive / negative pair
    uint64_t bmp, bmn;    // mass before them
    uint32_t tot_c;
    uint64_t tot_m;
};

__device__ SegPos segment_positions(const OwnSegs& o, HScratch& s)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t cp = o.cp[0] + o.cp[1], cn = o.cn[0] + o.cn[1];
    const uint64_t mp = o.mp[0] + o.mp[1], mn = o.mn[0] + o.mn[1];
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
        const bool in = lane < kHW;
        const uint32_t c1 = in ? s.wcp[lane] : 0u, c2 = in ? s.wcn[lane] : 0u;
        const uint64_t m1 = in ? s.wmp[lane] : 0u, m2 = in ? s.wmn[lane] : 0u;
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
        if (in) {
            s.wcp[lane] = a1 - c1;  // positive: the warps above this one
            s.wmp[lane] = b1 - m1;
            s.wcn[lane] = a2 - c2;  // negative: the warps below this one
            s.wmn[lane] = b2 - m2;
        }
        if (lane == 0) {
            s.tot_pc = a1;
            s.tot_pm = b1;
        }
        if (lane == kHW - 1) {
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

// The segment where the running count (BY_MASS false) or mass (true) in
// value order first reaches `need`: the thread that owns it records it.
// Exactly one segment qualifies when 0 < need <= total.
template <bool BY_MASS>
__device__ void claim_segment(const SegPos& p, const OwnSegs& o, uint64_t need, HScratch& s)
{
    const int t = threadIdx.x;
    constexpr int slot = BY_MASS ? 1 : 0;
    auto test = [&](uint32_t bc, uint64_t bm, uint32_t cnt, uint64_t mass, int seg) {
        const bool hit = BY_MASS ? (bm < need && need <= bm + mass && mass > 0)
                                 : (bc < need && need <= static_cast<uint64_t>(bc) + cnt);
        if (hit) {
            s.seg[slot] = seg;
            s.seg_c[slot] = bc;
            s.seg_m[slot] = bm;
        }
    };
    // Positive: segment 2t + 1 (larger magnitudes) comes before 2t.
    test(p.bcp, p.bmp, o.cp[1], o.mp[1], 2 * t + 1);
    test(p.bcp + o.cp[1], p.bmp + o.mp[1], o.cp[0], o.mp[0], 2 * t);
    // Negative: segment 2t (smaller magnitudes) comes before 2t + 1.
    test(p.bcn, p.bmn, o.cn[0], o.mn[0], kSegs + 2 * t);
    test(p.bcn + o.cn[0], p.bmn + o.mn[0], o.cn[1], o.mn[1], kSegs + 2 * t + 1);
}

// The table mode that holds segment seg (index + kSegs if negative) in full.
__device__ __forceinline__ int mode_of_seg(int seg)
{
    const bool neg = seg >= kSegs;
    const int j = neg ? seg - kSegs : seg;
    return (neg ? kQ2 : kQ0) + (j >= kSegs / 2 ? 1 : 0);
}

// Warp 0: walks the claimed segment, one magnitude per lane in value order,
// to the first value where the running count or mass reaches `need`; records
// that value and the mass of its upper set. The table (mode MODE) must hold
// the segment.
template <int MODE, bool BY_MASS>
__device__ void walk_segment(const uint32_t* win, float c, float mref, uint64_t need, HScratch& s)
{
    const uint32_t lane = threadIdx.x & 31u;
    constexpr int slot = BY_MASS ? 1 : 0;
    const int seg = s.seg[slot];
    const bool pos = seg < kSegs;
    const uint32_t j = static_cast<uint32_t>(pos ? seg : seg - kSegs);
    // Positive values descend with the magnitude, negative ones ascend.
    const uint32_t g = 32u * j + (pos ? 31u - lane : lane);
    uint32_t np = 0, nn = 0;
    if (SV_IN_RANGE(g - table_g0<MODE>(), kWin)) split_word<MODE>(win[g - table_g0<MODE>()], &np, &nn);
    else s.check = kFlagIndex;
    const uint32_t n = pos ? np : nn;
    const float v = pos ? __uint_as_float(g << 16) : -__uint_as_float(g << 16);
    const uint64_t m = n ? mass_n(n, v, c, mref) : 0u;
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
    const bool hit = BY_MASS ? (s.seg_m[slot] + cm >= need) : (s.seg_c[slot] + cc >= need);
    const unsigned b = __ballot_sync(0xFFFFFFFFu, hit);
    if (b != 0u && lane == static_cast<uint32_t>(__ffs(b) - 1)) {
        s.tau = v == 0.0f ? 0.0f : v;
        s.through = s.seg_m[slot] + cm;
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

// ---------------------------------------------------------------------------
// Selection on the packed window (every row whose counts did not wrap)
// ---------------------------------------------------------------------------
// How a selection ended: thresholds found; count the row again with 32-bit
// counts; no crossing found (impossible with exact integer sums); (a scan)
// scan again.
enum { kSelOk = 0, kSelRecount = 1, kSelFail = 2, kSelAgain = 3 };

// Sum over the CTA of a count and a mass; every thread gets them. Its slots
// are read again only after the next row's barriers.
__device__ void block_sum2(uint32_t* c, uint64_t* m, HScratch& s)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t x = __reduce_add_sync(0xFFFFFFFFu, *c);
    uint64_t y = *m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) y += __shfl_xor_sync(0xFFFFFFFFu, y, off);
    if (lane == 0) {
        s.sum_c[w] = x;
        s.sum_m[w] = y;
    }
    __syncthreads();
    x = lane < kHW ? s.sum_c[lane] : 0u;
    y = lane < kHW ? s.sum_m[lane] : 0u;
    x = __reduce_add_sync(0xFFFFFFFFu, x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) y += __shfl_xor_sync(0xFFFFFFFFu, y, off);
    *c = x;
    *m = y;
}

// The count of every element and the row's whole mass, from the packed
// window and its two outer words: below the window (|x| < 2^-64) the mass of
// 0 each, above it none (x <= -2^64; a positive value there means a maximum
// of 2^64 or more, and such rows are counted again).
template <bool MASS>
__device__ void window_totals(const uint32_t* win, float c, float mref, uint32_t* cnt,
                              uint64_t* mass, HScratch& s)
{
    const uint32_t t = threadIdx.x, lane = t & 31u, w = t >> 5;
    const uint4* w4 = reinterpret_cast<const uint4*>(win);
    // Warp w takes blocks of 128 consecutive words, w, w + 16, ...: the words
    // present cluster (a row's values fill a few binades), so most blocks are
    // skipped whole and a dense one keeps all its lanes busy.
    constexpr int kBlocks = kWin / 128 / kHW;  // per warp
    constexpr int kBatch = 4;
    uint32_t n = 0;
    uint64_t m = 0;
    for (int i0 = 0; i0 < kBlocks; i0 += kBatch) {
        uint4 q[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) q[i] = w4[32u * (w + kHW * (i0 + i)) + lane];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t ws[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
            n += (ws[0] & 0xFFFFu) + (ws[0] >> 16) + (ws[1] & 0xFFFFu) + (ws[1] >> 16) +
                 (ws[2] & 0xFFFFu) + (ws[2] >> 16) + (ws[3] & 0xFFFFu) + (ws[3] >> 16);
            if (!MASS || !__any_sync(0xFFFFFFFFu, (ws[0] | ws[1] | ws[2] | ws[3]) != 0u)) continue;
            const uint32_t g4 = kG0 + 4u * (32u * (w + kHW * static_cast<uint32_t>(i0 + i)) + lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t np = ws[k] & 0xFFFFu, nn = ws[k] >> 16;
                const float v = __uint_as_float((g4 + k) << 16);
                if (np) m += mass_n(np, v, c, mref);
                if (nn) m += mass_n(nn, -v, c, mref);
            }
        }
    }
    if (t == 0) {
        const uint32_t lo = win[-1], hi = win[kWin];
        const uint32_t nt = (lo & 0xFFFFu) + (lo >> 16);
        n += nt + (hi & 0xFFFFu) + (hi >> 16);
        if (MASS) m += mass_n(nt, 0.0f, c, mref);
    }
    block_sum2(&n, &m, s);
    *cnt = n;
    *mass = m;
}

// The packed window's values in value order, from the row maximum down:
// positions [0, np) the positive magnitudes from the maximum's down to the
// window's first; then, if any value can lie there, the word below the
// window (|x| < 2^-64, both signs); then the negative magnitudes from i0
// (the maximum's, when the maximum is negative) up; then the word above it.
struct DownSeq {
    int np;
    int tiny;   // 1 when the word below the window has a position
    int i0;
    int n;      // number of positions
};

__device__ __forceinline__ DownSeq down_seq(float mx)
{
    DownSeq d;
    const int gm = static_cast<int>((__float_as_uint(mx) >> 16) & 0x7FFFu);
    const bool neg = __float_as_uint(mx) >> 31;
    const bool in = gm >= static_cast<int>(kG0);  // |mx| >= 2^-64 (and < 2^64: checked)
    d.np = !neg && in ? gm - static_cast<int>(kG0) + 1 : 0;
    d.tiny = neg && in ? 0 : 1;
    d.i0 = neg && in ? gm - static_cast<int>(kG0) : 0;
    d.n = d.np + d.tiny + (kWin - d.i0) + 1;
    return d;
}

// Finds, by a block-wide scan of 512 positions at a time in value order, the
// first value where the running count (KIND kByCount) or mass (kByMass)
// reaches `need` (0 < need <= total). Sets s.tau and s.through (the mass of
// the upper set of that value) and returns kSelOk; kSelRecount when the
// crossing falls on one of the outer words, whose values are not told apart.
// kByCountThenMass: top-k (need = k), then top-p (a fraction top_p of the
// top-k mass), which crosses at or above the top-k threshold; when it crosses
// in the same 512 positions their sums give it at once (s.tau, s.through the
// top-p results), otherwise kSelAgain (s.through the top-k mass).
enum { kByCount = 0, kByMass = 1, kByCountThenMass = 2 };

template <int KIND>
__device__ int scan_down(const uint32_t* win, const DownSeq& d, float c, float mref, uint64_t need,
                         float top_p, HScratch& s)
{
    constexpr bool BY_MASS = KIND == kByMass;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint64_t base_c = 0, base_m = 0;
    for (int p0 = 0; p0 < d.n; p0 += kHT) {
        const int p = p0 + t;
        uint32_t n = 0;
        uint64_t m = 0;
        float v = 0.0f;
        bool outer = false;
        if (p < d.np) {
            const int i = d.np - 1 - p;
            n = SV_IN_RANGE(i, kWin) ? win[i] & 0xFFFFu : (s.check = kFlagIndex, 0u);
            v = __uint_as_float((kG0 + static_cast<uint32_t>(i)) << 16);
            m = n ? mass_n(n, v, c, mref) : 0u;
        } else if (p < d.np + d.tiny) {
            const uint32_t lo = win[-1];
            n = (lo & 0xFFFFu) + (lo >> 16);
            m = mass_n(n, 0.0f, c, mref);
            outer = true;
        } else if (p < d.n) {
            const int i = d.i0 + (p - d.np - d.tiny);
            if (i < kWin) {
                n = SV_IN_RANGE(i, kWin) ? win[i] >> 16 : (s.check = kFlagIndex, 0u);
                v = -__uint_as_float((kG0 + static_cast<uint32_t>(i)) << 16);
                m = n ? mass_n(n, v, c, mref) : 0u;
            } else {
                n = win[kWin] >> 16;  // no mass
                outer = true;
            }
        }
        // Inclusive scan over the warp, then over the warps.
        uint32_t ic = n;
        uint64_t im = m;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t oc = __shfl_up_sync(0xFFFFFFFFu, ic, off);
            const uint64_t om = __shfl_up_sync(0xFFFFFFFFu, im, off);
            if (lane >= off) {
                ic += oc;
                im += om;
            }
        }
        if (lane == 31) {
            s.wcp[w] = ic;
            s.wmp[w] = im;
        }
        __syncthreads();
        // Lane l holds warp l's totals; an inclusive scan over them gives
        // what lies before this warp (lane w - 1) and the chunk's total.
        uint32_t xc = lane < kHW ? s.wcp[lane] : 0u;
        uint64_t xm = lane < kHW ? s.wmp[lane] : 0u;
#pragma unroll
        for (int off = 1; off < kHW; off <<= 1) {
            const uint32_t oc = __shfl_up_sync(0xFFFFFFFFu, xc, off);
            const uint64_t om = __shfl_up_sync(0xFFFFFFFFu, xm, off);
            if (lane >= off) {
                xc += oc;
                xm += om;
            }
        }
        const uint32_t pc = w > 0 ? __shfl_sync(0xFFFFFFFFu, xc, w - 1) : 0u;
        const uint64_t pm = w > 0 ? __shfl_sync(0xFFFFFFFFu, xm, w - 1) : 0u;
        const uint32_t tc = __shfl_sync(0xFFFFFFFFu, xc, kHW - 1);
        const uint64_t tm = __shfl_sync(0xFFFFFFFFu, xm, kHW - 1);
        const uint64_t cc = base_c + pc + ic, cm = base_m + pm + im;
        const bool hit = BY_MASS ? (m > 0 && cm >= need && cm - m < need)
                                 : (n > 0 && cc >= need && cc - n < need);
        if (hit) {
            s.tau = v == 0.0f ? 0.0f : v;
            s.through = cm;
            s.found = outer ? 2 : 1;
        }
        __syncthreads();
        if (KIND == kByCountThenMass && s.found == 1) {
            // The top-p target, and whether it is crossed in this chunk.
            const uint64_t target = ceil_frac(top_p, s.through);
            if (base_m >= target) {
                s.found = 3;  // crossed before this chunk: a second scan
            } else {
                __syncthreads();  // every thread has read s.through and s.found
                if (m > 0 && cm >= target && cm - m < target) {
                    s.tau = v == 0.0f ? 0.0f : v;
                    s.through = cm;
                    s.found = outer ? 2 : 1;
                }
                __syncthreads();
            }
        }
        if (s.found != 0) break;
        base_c += tc;
        base_m += tm;
    }
    const int f = s.found;
    __syncthreads();  // every thread has read s.found before the next scan resets it
    if (t == 0) s.found = 0;
    return f == 1 ? kSelOk : (f == 2 ? kSelRecount : (f == 3 ? kSelAgain : kSelFail));
}

// Per-row constants of the selection.
struct CutK {
    bool tk, tp;
    uint64_t k;
    float top_p;
    float c;
};

// Everything a row's selection needs from the kernel.
struct RowCtx {
    const uint8_t* row;
    int64_t V;
    uint8_t* tabmem;
    uint32_t* win;        // window word 0 (generic pointer)
    uint32_t win_s;       // its shared address
    float mref;
};

// The thresholds of a row counted again with 32-bit counts; every thread
// calls it. The table (a quarter, *mode_now) is counted again for the quarter
// that holds each claimed segment. kSelFail if no segment holds a crossing
// (impossible with exact integer sums; the row is reported as failed rather
// than read out of range).
__device__ int select_row(const RowCtx& R, const CutK& P, const SegPos& pos, const OwnSegs& o,
                          int* mode_now, HScratch& s, float* tau, uint64_t* kept)
{
    // The claim slots were reset before the segment positions were taken
    // (whose barriers order that before these writes).
    auto claim = [&](bool by_mass, uint64_t need) -> int {
        if (by_mass) claim_segment<true>(pos, o, need, s);
        else claim_segment<false>(pos, o, need, s);
        __syncthreads();
        const int seg = s.seg[by_mass ? 1 : 0];
        if (seg < 0) return kSelFail;
        if (!SV_IN_RANGE(seg, 2 * kSegs)) {
            s.check = kFlagIndex;
            return kSelFail;
        }
        const int want = mode_of_seg(seg);
        if (want != *mode_now) {
            zero_table(R.tabmem);
            __syncthreads();
            switch (want) {
            case kQ0: count_row<kQ0>(R.row, R.V, R.win_s); break;
            case kQ1: count_row<kQ1>(R.row, R.V, R.win_s); break;
            case kQ2: count_row<kQ2>(R.row, R.V, R.win_s); break;
            default: count_row<kQ3>(R.row, R.V, R.win_s); break;
            }
            __syncthreads();
            *mode_now = want;
        }
        return kSelOk;
    };
    auto walk = [&](bool by_mass, uint64_t need) {
        if (threadIdx.x < 32) {
            switch (*mode_now) {
            case kQ0:
                if (by_mass) walk_segment<kQ0, true>(R.win, P.c, R.mref, need, s);
                else walk_segment<kQ0, false>(R.win, P.c, R.mref, need, s);
                break;
            case kQ1:
                if (by_mass) walk_segment<kQ1, true>(R.win, P.c, R.mref, need, s);
                else walk_segment<kQ1, false>(R.win, P.c, R.mref, need, s);
                break;
            case kQ2:
                if (by_mass) walk_segment<kQ2, true>(R.win, P.c, R.mref, need, s);
                else walk_segment<kQ2, false>(R.win, P.c, R.mref, need, s);
                break;
            default:
                if (by_mass) walk_segment<kQ3, true>(R.win, P.c, R.mref, need, s);
                else walk_segment<kQ3, false>(R.win, P.c, R.mref, need, s);
                break;
            }
        }
        __syncthreads();
    };

    float t_val = __uint_as_float(kF32NegInfBits);
    uint64_t mass_k = pos.tot_m;
    if (P.tk) {
        const int st = claim(false, P.k);
        if (st != kSelOk) return st;
        walk(false, P.k);
        t_val = s.tau;
        mass_k = s.through;
    }
    if (P.tp) {
        const uint64_t target = ceil_frac(P.top_p, mass_k);
        const int st = claim(true, target);
        if (st != kSelOk) return st;
        walk(true, target);
        t_val = s.tau;
        *kept = s.through;
    } else {
        *kept = mass_k;
    }
    *tau = t_val;
    return kSelOk;
}

// The thresholds of a row counted in the packed window without a wrap.
__device__ int fast_select(const uint32_t* win, const CutK& P, float mx, float mref, uint64_t tot_m,
                           HScratch& s, float* tau, uint64_t* kept)
{
    const DownSeq d = down_seq(mx);
    if (P.tk && P.tp) {
        int st = scan_down<kByCountThenMass>(win, d, P.c, mref, P.k, P.top_p, s);
        if (st == kSelAgain)
            st = scan_down<kByMass>(win, d, P.c, mref, ceil_frac(P.top_p, s.through), 0.f, s);
        if (st != kSelOk) return st;
    } else if (P.tk) {
        const int st = scan_down<kByCount>(win, d, P.c, mref, P.k, 0.f, s);
        if (st != kSelOk) return st;
    } else {
        const int st = scan_down<kByMass>(win, d, P.c, mref, ceil_frac(P.top_p, tot_m), 0.f, s);
        if (st != kSelOk) return st;
    }
    *tau = s.tau;
    *kept = s.through;
    return kSelOk;
}

__device__ void fail_rows(const FilterArgs& a, int flags)
{
    if (threadIdx.x != 0) return;
    for (int64_t r = blockIdx.x; r < a.g.rows; r += gridDim.x) a.rows[r] = FiltRow{0.f, 0.f, 0.f, flags};
}

__global__ void __launch_bounds__(kHT, 2) hist_kernel(const __grid_constant__ FilterArgs a)
{
    extern __shared__ __align__(16) uint8_t hsm[];
    __shared__ HScratch s;
    const int t = threadIdx.x;
    const int64_t V = a.g.V;
    uint32_t* win = reinterpret_cast<uint32_t*>(hsm + 16);
    const SegArrays A{reinterpret_cast<uint32_t*>(hsm + kTabBytes),
                      reinterpret_cast<uint64_t*>(hsm + kTabBytes + kSegs * 4),
                      reinterpret_cast<uint32_t*>(hsm + kTabBytes + kSegs * 12),
                      reinterpret_cast<uint64_t*>(hsm + kTabBytes + kSegs * 16)};
    RowCtx R{nullptr, V, hsm, win, smem_addr(win), 0.f};
    if (t == 0) s.found = 0;
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
        R.row = r < a.g.rows_t ? a.target + r * V * 2 : a.draft + (r - a.g.rows_t) * V * 2;
        const RowVecs rv = row_vecs(R.row, V);
        uint4 u[kHU];
        load_batch(rv, 0, u);  // in flight while the table is cleared
        if (t == 0) s.check = 0;  // thread 0 wrote the previous row's result
        __syncthreads();       // the previous row is done with the table
        zero_table(hsm);
        __syncthreads();
        float tm;
        count_vecs<kPacked, true>(rv, R.win_s, u, &tm);
        const float mx = block_max(tm, s);  // its barriers also order the counts before the sweep
        if (!(mx > __uint_as_float(kF32NegInfBits)) || !(mx < __uint_as_float(0x7F800000u))) {
            // NaN or +inf in the row, or no finite logit.
            if (t == 0) a.rows[r] = FiltRow{0.f, 0.f, 0.f, kFlagNonFinite};
            continue;
        }
        R.mref = ceilf(mx * P.c);
        // This thread's segments 2t, 2t + 1 of each sign (32-bit counts).
        auto own = [&]() {
            __syncthreads();  // the segment arrays are written
            if (t == 0) {
                s.seg[0] = -1;
                s.seg[1] = -1;
            }
            OwnSegs o;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                o.cp[i] = A.cp[2 * t + i];
                o.mp[i] = A.mp[2 * t + i];
                o.cn[i] = A.cn[2 * t + i];
                o.mn[i] = A.mn[2 * t + i];
            }
            return o;
        };
        uint32_t tot_c;
        uint64_t tot_m;
        // The whole mass is the top-p target's base when top-k is off.
        if (P.tp && !P.tk) window_totals<true>(win, P.c, R.mref, &tot_c, &tot_m, s);
        else window_totals<false>(win, P.c, R.mref, &tot_c, &tot_m, s);
        float tau = 0.f;
        uint64_t kept = 0;
        int st = kSelRecount;
        // A wrapped 16-bit count shows as counts short of V.
        if (tot_c == static_cast<uint64_t>(V) && mx < 18446744073709551616.0f)
            st = fast_select(win, P, mx, R.mref, tot_m, s, &tau, &kept);
        if (st == kSelRecount) {
            // Count again: 32 bits per magnitude, a quarter per read.
            __syncthreads();
            zero_table(hsm);
            __syncthreads();
            count_row<kQ0>(R.row, V, R.win_s);
            __syncthreads();
            segment_sums<kQ0>(win, P.c, R.mref, A);
            __syncthreads();
            zero_table(hsm);
            __syncthreads();
            count_row<kQ1>(R.row, V, R.win_s);
            __syncthreads();
            segment_sums<kQ1>(win, P.c, R.mref, A);
            __syncthreads();
            zero_table(hsm);
            __syncthreads();
            count_row<kQ2>(R.row, V, R.win_s);
            __syncthreads();
            segment_sums<kQ2>(win, P.c, R.mref, A);
            __syncthreads();
            zero_table(hsm);
            __syncthreads();
            count_row<kQ3>(R.row, V, R.win_s);
            __syncthreads();
            segment_sums<kQ3>(win, P.c, R.mref, A);
            const OwnSegs o = own();
            const SegPos pos = segment_positions(o, s);
            int mode_now = kQ3;
            st = pos.tot_c == static_cast<uint64_t>(V) ? select_row(R, P, pos, o, &mode_now, s, &tau, &kept)
                                                        : kSelFail;
        }
        if (t == 0) {
            const float l = log2f(__ull2float_rn(kept)) - 40.0f;
            a.rows[r] = s.check != 0                 ? FiltRow{0.f, 0.f, 0.f, s.check}
                        : st == kSelOk && kept > 0 ? FiltRow{R.mref, l, tau, 0}
                                                   : FiltRow{0.f, 0.f, 0.f, kFlagNonFinite};
        }
    }
}

}  // namespace

cudaError_t launch_hist(const FilterArgs& a, int sms, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHSmem);
    if (e != cudaSuccess) return e;
    const int64_t cap = 2 * static_cast<int64_t>(sms);
    const int64_t grid = a.g.rows < cap ? a.g.rows : cap;
    if (grid <= 0) return cudaSuccess;
    // The first kernel of a call: launched without programmatic dependent
    // launch, so the caller's earlier work on the stream (the logits) is
    // complete and visible before the first read.
    return launch_dependent(false, hist_kernel, dim3(static_cast<unsigned>(grid)), dim3(kHT),
                            static_cast<size_t>(kHSmem), s, a);
}

}  // namespace sv
