// row_stats.cu -- pass 1: per-row softmax normalisers (or argmaxes) of the
// target and draft logits, read from HBM exactly once.
//
// What it computes ("Как работает speculative decoding на уровне логитов..."
// (aivaro.ru) §9 and "Speculative decoding" (aihero.vn), temperature
// paragraph): for every target row and every draft row, the log-sum-exp of
// logits / T, which turns each raw logit into log p or log q. In greedy mode
// ("Speculative decoding" (aihero.vn), "Cùng phân bố không có nghĩa cùng
// chuỗi") it computes instead the lowest index of each target row's maximum.
//
// Design. The rows of both tensors form one row space [target | draft], cut
// into fixed tiles of kRowTileBytes. The grid is the number of SMs times the
// resident CTAs per SM; CTA g takes the contiguous tile range
// [g*T/G, (g+1)*T/G), so every CTA streams the same number of bytes (within
// one tile) whatever the row length. Per CTA one producer lane moves tiles
// with 1-D bulk copies (cp.async.bulk, the TMA engine's untiled form) into a
// kRowStages-deep ring of shared-memory buffers guarded by full/empty
// mbarriers; kRowConsumerWarps warps read the tiles with 16-byte shared loads.
// Each consumer warp keeps its own running state and writes one Partial per
// row segment it saw, so consumers never wait on each other: the only
// synchronisation after start-up is the ring's mbarriers, and every wait on
// them is bounded.
//
// Numerics (sampling). Logits are scaled by c = log2(e)/T and summed as
// 2^(x*c - m) on the SFU. The reference exponent m is an integer (the ceiling
// of the largest scaled logit seen so far), so every rescale is an exact power
// of two. Per tile a thread adds <= 32 terms in four float accumulators, then
// folds the tile sum into a float pair (two-sum), keeping the running sum's
// rounding error. Warps combine their lanes as float pairs (no float64: GB300
// runs it at a small fraction of the float32 rate).
#include <climits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kNC = kRowConsumerWarps * 32;          // consumer threads
constexpr int kVecPerTile = kRowTileBytes / 16;      // 16-byte vectors per tile
constexpr int kVPT = kVecPerTile / kNC;              // vectors per consumer thread
static_assert(kVecPerTile % kNC == 0, "tile must split evenly over consumers");
constexpr int kSampleMode = 0;
constexpr int kGreedyMode = 1;

__device__ __forceinline__ const uint8_t* align_down16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15));
}
__device__ __forceinline__ const uint8_t* align_up16(const uint8_t* p)
{
    return reinterpret_cast<const uint8_t*>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
}

// Walks the tiles of a CTA's range in order, without divisions per tile.
struct Cursor {
    int64_t row;             // pass-1 row in the launch's row space
    int64_t k;               // tile index within the row
    int64_t n;               // sequences in the row space
    int64_t goff;            // token index of the row's first element (a shard row's offset)
    int64_t ridx;            // row index within its tensor ([B, K+1] target or [B, K] draft)
    int tensor;              // 0 target, 1 draft
    const uint8_t* rowp;     // first byte of the row (one-tensor rows)
    const uint8_t* tend;     // 16-byte-aligned end of the row's tensor
};

// Pass-1 row `row`: logical row R = row / RS of the row space
// [n * nt target rows | n * nd draft rows] (in each part sequence s of the map
// contributes its positions p0, p0 + 1, ... in order), and with RS = G shard
// rows per logical row, shard row % G of it. With the identity map and
// RS = 1 this is the plain concatenation [target rows | draft rows].
template <int ES>
__device__ __forceinline__ void cursor_row(Cursor& c, const RowStatsArgs& a, int64_t row)
{
    const Geometry& g = a.g;
    const RowMap& m = a.map;
    const int64_t RS = g.row_shards;
    c.row = row;
    const int64_t row_bytes = g.row_len * ES;
    if (row >= c.n * (m.nt + m.nd) * RS) {
        // One past the last row (the cursor steps here after the last tile):
        // never copied from, and the map has no entry for it.
        c.rowp = a.target;
        c.tend = a.target;
        c.goff = 0;
        c.ridx = 0;
        c.tensor = 0;
        return;
    }
    const int64_t lr = row / RS;
    const int gi = static_cast<int>(row - lr * RS);
    c.goff = gi * g.row_len;
    const int64_t nt_rows = c.n * m.nt;
    if (lr < nt_rows) {
        const int64_t sq = lr / m.nt, i = m.p0 + (lr - sq * m.nt);
        const int64_t b = m.active != nullptr ? m.active[sq] : sq;
        c.tensor = 0;
        c.ridx = b * (g.K + 1) + i;
        c.rowp = a.sh.t[gi] + c.ridx * row_bytes;
        c.tend = align_down16(a.sh.t[gi] + g.rows_t * row_bytes);
    } else {
        const int64_t r = lr - nt_rows;
        const int64_t sq = r / m.nd, i = m.p0 + (r - sq * m.nd);
        const int64_t b = m.active != nullptr ? m.active[sq] : sq;
        c.tensor = 1;
        c.ridx = b * g.K + i;
        c.rowp = a.sh.d[gi] + c.ridx * row_bytes;
        c.tend = align_down16(a.sh.d[gi] + g.B * g.K * row_bytes);
    }
}

template <int ES>
__device__ __forceinline__ void cursor_next(Cursor& c, const RowStatsArgs& a)
{
    if (++c.k == a.g.tiles_per_row) {
        c.k = 0;
        cursor_row<ES>(c, a, c.row + 1);
    }
}

// Where one tile's bytes come from and how they sit in its stage buffer.
// The buffer holds the 16-byte-aligned range [a0, a0 + 16 nv) that covers the
// tile's bytes [s, e); bytes outside [s, e) are masked by the consumers.
struct Span {
    const uint8_t* a0;   // aligned start of the buffer's range
    uint32_t bulk;       // bytes the bulk copy moves from a0
    const uint8_t* tail; // bytes [tail, e) are loaded one element at a time
    const uint8_t* e;    // end of the tile
    int32_t nv;          // vectors in the buffer
    int32_t head;        // elements of vector 0 before the tile
    int32_t last;        // valid elements of vector nv - 1
    int64_t idx0;        // row index of vector 0's first element
};

// What consumers need to know about the tile in a stage. The producer, which
// computes the span anyway, writes it next to the data before its arrive.
struct TileRec {
    int32_t seg;      // row - first row of the CTA
    int32_t nv;       // vectors in the buffer
    int32_t head;     // elements of vector 0 before the tile
    int32_t last;     // valid elements of vector nv - 1
    long long idx0;   // row index of vector 0's first element
};

template <int ES>
__device__ __forceinline__ Span tile_span(const Cursor& c, const Geometry& g)
{
    Span sp;
    const int64_t e0 = c.k * g.tile_elems;
    const int64_t e1 = min(e0 + g.tile_elems, g.row_len);
    const uint8_t* s = c.rowp + e0 * ES;
    const uint8_t* e = c.rowp + e1 * ES;
    if (g.row_aligned) {
        // Rows, tiles and tensor ends on 16-byte boundaries: no cover, no
        // masks, no element-wise tail.
        sp.a0 = s;
        sp.bulk = static_cast<uint32_t>(e - s);
        sp.tail = e;
        sp.e = e;
        sp.nv = static_cast<int32_t>(sp.bulk >> 4);
        sp.head = 0;
        sp.last = 16 / ES;
        sp.idx0 = c.goff + e0;
        return sp;
    }
    sp.a0 = align_down16(s);
    const uint8_t* up = align_up16(e);
    const uint8_t* bend = up < c.tend ? up : c.tend;
    sp.bulk = bend > sp.a0 ? static_cast<uint32_t>(bend - sp.a0) : 0u;
    sp.tail = bend >= e ? e : (bend > s ? bend : s);
    sp.e = e;
    sp.nv = static_cast<int32_t>((e - sp.a0 + 15) >> 4);
    sp.head = static_cast<int32_t>((s - sp.a0) / ES);
    sp.last = static_cast<int32_t>((e - (sp.a0 + 16 * (sp.nv - 1))) / ES);
    sp.idx0 = c.goff + e0 - sp.head;
    return sp;
}

// Replace the elements of a 16-byte vector outside [lo, hi) by -inf.
template <int ES>
__device__ __forceinline__ void mask_vector(uint4& v, int lo, int hi)
{
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (ES == 2) {
#pragma unroll
        for (int el = 0; el < 8; ++el) {
            if (el < lo || el >= hi) {
                uint32_t& x = w[el >> 1];
                x = (el & 1) ? ((x & 0x0000FFFFu) | 0xFF800000u) : ((x & 0xFFFF0000u) | 0x0000FF80u);
            }
        }
    } else {
#pragma unroll
        for (int el = 0; el < 4; ++el)
            if (el < lo || el >= hi) w[el] = kF32NegInfBits;
    }
    v = make_uint4(w[0], w[1], w[2], w[3]);
}

template <int ES>
__device__ __forceinline__ void load_tile(uint4 (&v)[kVPT], const uint8_t* buf, const TileRec& sp,
                                          int tid, bool aligned)
{
    const uint32_t fill = ES == 2 ? kBf16NegInfPair : kF32NegInfBits;
#pragma unroll
    for (int q = 0; q < kVPT; ++q) {
        const int vi = tid + q * kNC;
        v[q] = vi < sp.nv ? ld_shared_v4(buf + 16 * vi) : make_uint4(fill, fill, fill, fill);
    }
    if (!aligned) {
#pragma unroll
        for (int q = 0; q < kVPT; ++q) {
            const int vi = tid + q * kNC;
            if (vi < sp.nv && (vi == 0 || vi == sp.nv - 1))
                mask_vector<ES>(v[q], vi == 0 ? sp.head : 0, vi == sp.nv - 1 ? sp.last : 16 / ES);
        }
    }
}

// Largest element of the thread's share of a tile (NaN if any is NaN).
template <int ES>
__device__ __forceinline__ float tile_max(const uint4 (&v)[kVPT])
{
    if (ES == 2) {
        uint32_t m = kBf16NegInfPair;
#pragma unroll
        for (int q = 0; q < kVPT; ++q) {
            m = bf16x2_max_nan(m, v[q].x);
            m = bf16x2_max_nan(m, v[q].y);
            m = bf16x2_max_nan(m, v[q].z);
            m = bf16x2_max_nan(m, v[q].w);
        }
        return fmax_nan(bf16_lo(m), bf16_hi(m));
    } else {
        float m0 = __uint_as_float(kF32NegInfBits), m1 = m0;
#pragma unroll
        for (int q = 0; q < kVPT; ++q) {
            m0 = fmax_nan(m0, __uint_as_float(v[q].x));
            m1 = fmax_nan(m1, __uint_as_float(v[q].y));
            m0 = fmax_nan(m0, __uint_as_float(v[q].z));
            m1 = fmax_nan(m1, __uint_as_float(v[q].w));
        }
        return fmax_nan(m0, m1);
    }
}

struct SampleState {
    float m;       // reference exponent (integer-valued), -inf before any finite logit
    float s_hi;    // running sum of 2^(x c - m) as hi + lo
    float s_lo;
    int flags;
    __device__ __forceinline__ void reset()
    {
        m = __uint_as_float(kF32NegInfBits);
        s_hi = 0.f;
        s_lo = 0.f;
        flags = 0;
    }
};

struct GreedyState {
    float best;    // largest raw logit seen
    int idx;       // its lowest row index, INT_MAX if nothing beat -inf
    int flags;
    __device__ __forceinline__ void reset()
    {
        best = __uint_as_float(kF32NegInfBits);
        idx = INT_MAX;
        flags = 0;
    }
};

template <int ES>
__device__ __forceinline__ void accumulate_tile(SampleState& st, const uint4 (&v)[kVPT], float c)
{
    const float tmax = tile_max<ES>(v);
    if (tmax != tmax || tmax == __uint_as_float(0x7F800000u)) {  // NaN or +inf
        st.flags |= kFlagNonFinite;
        return;
    }
    const float mt = ceilf(tmax * c);
    if (mt > st.m) {
        const float sc = pow2_neg_int(st.m - mt);
        st.s_hi *= sc;
        st.s_lo *= sc;
        st.m = mt;
    }
    if (st.m == __uint_as_float(kF32NegInfBits)) return;  // only -inf so far
    const float nm = -st.m;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int q = 0; q < kVPT; ++q) {
        if (ES == 2) {
            a0 += ex2(fmaf(bf16_lo(v[q].x), c, nm));
            a1 += ex2(fmaf(bf16_hi(v[q].x), c, nm));
            a2 += ex2(fmaf(bf16_lo(v[q].y), c, nm));
            a3 += ex2(fmaf(bf16_hi(v[q].y), c, nm));
            a0 += ex2(fmaf(bf16_lo(v[q].z), c, nm));
            a1 += ex2(fmaf(bf16_hi(v[q].z), c, nm));
            a2 += ex2(fmaf(bf16_lo(v[q].w), c, nm));
            a3 += ex2(fmaf(bf16_hi(v[q].w), c, nm));
        } else {
            a0 += ex2(fmaf(__uint_as_float(v[q].x), c, nm));
            a1 += ex2(fmaf(__uint_as_float(v[q].y), c, nm));
            a2 += ex2(fmaf(__uint_as_float(v[q].z), c, nm));
            a3 += ex2(fmaf(__uint_as_float(v[q].w), c, nm));
        }
    }
    two_sum_acc(st.s_hi, st.s_lo, (a0 + a1) + (a2 + a3));
}

template <int ES>
__device__ __forceinline__ void argmax_tile(GreedyState& st, const uint4 (&v)[kVPT],
                                            const TileRec& sp, int tid)
{
    const float tmax = tile_max<ES>(v);
    if (tmax != tmax) {
        st.flags |= kFlagNonFinite;
        return;
    }
    if (!(tmax > st.best)) return;
    // The tile beats the running best: find the first element equal to it, in
    // increasing index order (this thread's vectors ascend with q).
    int found = INT_MAX;
#pragma unroll
    for (int q = 0; q < kVPT; ++q) {
        const int vi = tid + q * kNC;
        const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int el = 0; el < 16 / ES; ++el) {
            const float x = ES == 2 ? ((el & 1) ? bf16_hi(w[el >> 1]) : bf16_lo(w[el >> 1]))
                                    : __uint_as_float(w[el]);
            if (found == INT_MAX && x == tmax)
                found = static_cast<int>(sp.idx0 + static_cast<int64_t>(vi) * (16 / ES) + el);
        }
    }
    st.best = tmax;
    st.idx = found;
}

// Warp-reduce the lanes' states (float pairs, exact power-of-two rescales) and
// have lane 0 store the warp's Partial.
__device__ __forceinline__ void flush_sample(const SampleState& st, Partial* out, int lane)
{
    float m = st.m, hi = st.s_hi, lo = st.s_lo;
    int flags = st.flags;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xFFFFFFFFu, m, off);
        const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
        const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
        flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, off);
        merge_scaled(m, hi, lo, om, ohi, olo);
    }
    if (lane == 0) {
        Partial p;
        p.m = m;
        p.hi = hi;
        p.lo = lo;
        p.flags = flags;
        *out = p;
    }
}

__device__ __forceinline__ void flush_greedy(const GreedyState& st, Partial* out, int lane)
{
    float best = st.best;
    int idx = st.idx;
    int flags = st.flags;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, idx, off);
        flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, off);
        if (ob > best || (ob == best && oi < idx)) {
            best = ob;
            idx = oi;
        }
    }
    if (lane == 0) {
        Partial p;
        p.m = best;
        p.hi = __int_as_float(idx);
        p.lo = 0.f;
        p.flags = flags;
        *out = p;
    }
}

template <int ES, int MODE>
__global__ void __launch_bounds__(kRowThreads) row_stats_kernel(const __grid_constant__ RowStatsArgs a)
{
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t full_bar[kRowStages];
    __shared__ __align__(8) uint64_t empty_bar[kRowStages];
    __shared__ __align__(8) TileRec recs[kRowStages];
    __shared__ int abort_flag;

    const Geometry& g = a.g;
    const int cta = blockIdx.x;
    // Sequences in this launch's row space: all B, or (early exit) those the
    // previous scan left undecided, known once that scan has finished.
    int64_t nseq = g.B;
    if (a.map.count != nullptr) {
        pdl_wait();
        nseq = *a.map.count;
    }
    const int64_t tiles = map_rows(a.map, nseq) * g.row_shards * g.tiles_per_row;
    // CTAs in use: at most one per tile, so every range below is non-empty
    // (an early-exit phase can have fewer tiles than the launch has CTAs).
    const int64_t grid = tiles < g.grid ? tiles : g.grid;
    if (cta >= grid) return;
    const int64_t t_begin = static_cast<int64_t>(cta) * tiles / grid;
    const int64_t t_end = static_cast<int64_t>(cta + 1) * tiles / grid;
    const int64_t ntiles = t_end - t_begin;
    if (ntiles <= 0) return;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t row_first = t_begin / g.tiles_per_row;
    const int64_t row_last = (t_end - 1) / g.tiles_per_row;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRowStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kRowConsumerWarps);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    Cursor cur;
    cur.k = t_begin - row_first * g.tiles_per_row;
    cur.n = nseq;
    cursor_row<ES>(cur, a, row_first);

    if (warp == kRowConsumerWarps) {
        // ---------------- producer ----------------
        if (lane != 0) return;
        int64_t n = 0;
        if (a.gate != nullptr) {
            // Test hook: hold every copy until *gate != 0, bounded like every
            // other wait. Nothing sets it in the tests that use it, so the
            // consumers see the abort and mark their rows as timed out.
            const volatile int32_t* gate = a.gate;
            const long long t0 = clock64();
            while (*gate == 0) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    abort_flag = 1;
                    n = -1;
                    break;
                }
                __nanosleep(1000);
            }
            if (n < 0) return;  // no copy was issued
        }
        for (; n < ntiles; ++n) {
            const int stage = static_cast<int>(n % kRowStages);
            if (n >= kRowStages) {
                const uint32_t parity = static_cast<uint32_t>((n / kRowStages - 1) & 1);
                if (!mbar_wait_bounded(&empty_bar[stage], parity, &abort_flag)) {
                    abort_flag = 1;
                    break;
                }
            }
            const Span sp = tile_span<ES>(cur, g);
            uint8_t* dst = ring + static_cast<size_t>(stage) * kRowTileBytes;
            TileRec rec;
            rec.seg = static_cast<int32_t>(cur.row - row_first);
            rec.nv = sp.nv;
            rec.head = sp.head;
            rec.last = sp.last;
            rec.idx0 = sp.idx0;
            recs[stage] = rec;  // published by the arrive below (release)
            // Bytes the bulk copy cannot take (the last <16 bytes of a tensor
            // whose size is not a multiple of 16) go through plain loads.
            for (const uint8_t* p = sp.tail; p < sp.e; p += ES) {
                if (ES == 2)
                    *reinterpret_cast<uint16_t*>(dst + (p - sp.a0)) =
                        __ldg(reinterpret_cast<const unsigned short*>(p));
                else
                    *reinterpret_cast<uint32_t*>(dst + (p - sp.a0)) =
                        __ldg(reinterpret_cast<const unsigned int*>(p));
            }
            if (g.shards > 1 && g.row_shards == 1) {
                // A logical-row tile [e0, e1) of sharded logits: one bulk copy
                // per shard it overlaps, each landing at its place in the
                // stage. Shard widths fill whole 16-byte vectors, so every
                // piece starts and ends on a 16-byte boundary.
                const int64_t e0 = cur.k * g.tile_elems;
                const int64_t e1 = min(e0 + g.tile_elems, g.row_len);
                const int64_t Vs = g.shard_len;
                mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>((e1 - e0) * ES));
                for (int64_t gi = e0 / Vs; gi * Vs < e1; ++gi) {
                    const int64_t p0 = max(e0, gi * Vs), p1 = min(e1, (gi + 1) * Vs);
                    const uint8_t* base = cur.tensor == 0 ? a.sh.t[gi] : a.sh.d[gi];
                    bulk_copy_g2s(dst + (p0 - e0) * ES, base + (cur.ridx * Vs + (p0 - gi * Vs)) * ES,
                                  static_cast<uint32_t>((p1 - p0) * ES), &full_bar[stage]);
                }
            } else if (sp.bulk > 0) {
                mbar_arrive_expect_tx(&full_bar[stage], sp.bulk);
                bulk_copy_g2s(dst, sp.a0, sp.bulk, &full_bar[stage]);
            } else {
                mbar_arrive(&full_bar[stage]);
            }
            cursor_next<ES>(cur, a);
        }
        if (n < ntiles) {
            // Gave up: let the copies already issued land before the CTA exits.
            for (int64_t m = (n > kRowStages ? n - kRowStages : 0); m < n; ++m)
                mbar_wait_bounded(&full_bar[m % kRowStages],
                                  static_cast<uint32_t>((m / kRowStages) & 1), nullptr);
        }
        return;
    }

    // ---------------- consumers ----------------
    const int tid = threadIdx.x;  // 0 .. kNC-1
    const bool aligned = g.row_aligned != 0;
    Partial* my_partials =
        a.partials + static_cast<int64_t>(cta) * g.maxseg * kRowConsumerWarps + warp;
    SampleState ss;
    GreedyState gs;
    ss.reset();
    gs.reset();
    int seg = 0;  // the row segment being reduced (row - row_first)
    int64_t n = 0;
    int stage = 0;
    uint32_t parity = 0;
    for (; n < ntiles; ++n) {
        if (!mbar_wait_bounded(&full_bar[stage], parity, &abort_flag)) {
            abort_flag = 1;
            break;
        }
        TileRec sp = recs[stage];
        if (!SV_IN_RANGE(sp.seg, g.maxseg)) {
            // A tile record outside this CTA's segments: its elements are
            // skipped and the segment being reduced is reported.
            ss.flags |= kFlagIndex;
            gs.flags |= kFlagIndex;
            sp.seg = seg;
            sp.nv = 0;
        }
        if (sp.seg != seg) {
            Partial* out = my_partials + static_cast<int64_t>(seg) * kRowConsumerWarps;
            if (MODE == kSampleMode) {
                flush_sample(ss, out, lane);
                ss.reset();
            } else {
                flush_greedy(gs, out, lane);
                gs.reset();
            }
            seg = sp.seg;
        }
        uint4 v[kVPT];
        load_tile<ES>(v, ring + static_cast<size_t>(stage) * kRowTileBytes, sp, tid, aligned);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
        if (MODE == kSampleMode)
            accumulate_tile<ES>(ss, v, a.c);
        else
            argmax_tile<ES>(gs, v, sp, tid);
        if (++stage == kRowStages) {
            stage = 0;
            parity ^= 1u;
        }
    }
    // The scan may start launching now; it waits for this grid to finish.
    if (tid == 0) pdl_trigger();
    if (n == ntiles) {
        Partial* out = my_partials + static_cast<int64_t>(seg) * kRowConsumerWarps;
        if (MODE == kSampleMode)
            flush_sample(ss, out, lane);
        else
            flush_greedy(gs, out, lane);
    } else if (lane == 0) {
        // Timed out: mark this warp's remaining segments so the scan rejects them.
        for (int64_t r = row_first + seg; r <= row_last; ++r) {
            Partial p;
            p.m = __uint_as_float(kF32NegInfBits);
            p.hi = 0.f;
            p.lo = 0.f;
            p.flags = kFlagTimeout;
            my_partials[(r - row_first) * kRowConsumerWarps] = p;
        }
    }
}

template <int ES, int MODE>
cudaError_t launch_one(const RowStatsArgs& a, cudaStream_t s)
{
    auto* k = row_stats_kernel<ES, MODE>;
    const int smem = kRowStages * kRowTileBytes;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // The first pass of a call starts in plain stream order; an early-exit
    // phase after the first is chained to the scan it reads the list of.
    const bool pdl = a.g.pdl != 0 && a.map.count != nullptr;
    return launch_dependent(pdl, k, dim3(static_cast<unsigned>(a.g.grid)), dim3(kRowThreads),
                            static_cast<size_t>(smem), s, a);
}

template <int ES, int MODE>
cudaError_t occupancy_one(int* blocks)
{
    auto* k = row_stats_kernel<ES, MODE>;
    const int smem = kRowStages * kRowTileBytes;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k, kRowThreads, smem);
}

}  // namespace

cudaError_t launch_row_stats(const RowStatsArgs& a, cudaStream_t s)
{
    if (a.g.es == 2)
        return a.g.mode == kSampleMode ? launch_one<2, kSampleMode>(a, s)
                                       : launch_one<2, kGreedyMode>(a, s);
    return a.g.mode == kSampleMode ? launch_one<4, kSampleMode>(a, s)
                                   : launch_one<4, kGreedyMode>(a, s);
}

cudaError_t row_stats_blocks_per_sm(int es, int mode, int* blocks)
{
    if (es == 2)
        return mode == kSampleMode ? occupancy_one<2, kSampleMode>(blocks)
                                   : occupancy_one<2, kGreedyMode>(blocks);
    return mode == kSampleMode ? occupancy_one<4, kSampleMode>(blocks)
                               : occupancy_one<4, kGreedyMode>(blocks);
}

}  // namespace sv
