// lmhead.cu -- the LM head on the 5th-generation tensor cores: logits =
// hidden [R, D] x W[V, D]^T in bfloat16 with float32 accumulation.
//
// What it computes: the per-position logit vectors that "Как работает
// speculative decoding на уровне логитов..." (aivaro.ru) §4 and §5 step 1 take
// as given, made the way a language model's output layer makes them (h W^T).
// In the statistics mode the epilogue reduces each 256-column tile of a row
// to its part of the row's softmax normaliser at temperature T (§9 of the same
// page, "Speculative decoding" (aihero.vn) temperature paragraph), or, greedy,
// to the tile's maximum and lowest arg-max column, and keeps the draft token's
// logit; the logits themselves never reach HBM.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//  * warp 0 (one lane): TMA producer. Each k-block is a 128 x 64 tile of the
//    hidden states and a 256 x 64 tile of the weights (64 bf16 = 128 bytes of
//    K, 128-byte swizzle), loaded by cp.async.bulk.tensor into a 4-stage ring.
//  * warp 1: allocates 512 TMEM columns (two 128 x 256 float32 accumulators)
//    and, from one lane, issues tcgen05.mma (M = 128, N = 256, K = 16, four per
//    k-block); tcgen05.commit frees each ring stage when its MMAs complete and
//    signals a finished accumulator.
//  * warps 2..5: the epilogue. Each warp reads its 32 TMEM lanes (rows) with
//    tcgen05.ld, 32 columns at a time, while the MMA warp fills the other
//    accumulator.
// Tiles are ordered vocabulary-major, so the CTAs working at one time share
// the same weight tile through L2 and the hidden states stay resident.
// Every mbarrier wait is bounded; a wait that runs out sets the error word and
// the CTA winds down (TMEM is always released).
#include <cuda.h>

#include "sv_device.cuh"
#include "sv_stages.h"

namespace sv {
namespace {

constexpr int kBM = 128;              // rows of hidden states per tile (TMEM lanes)
constexpr int kBN = 256;              // vocabulary columns per tile (TMEM columns)
constexpr int kBK = 64;               // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUK = 16;               // K per tcgen05.mma (kind::f16)
constexpr int kStagesL = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kLmThreads = 192;
constexpr int kTmemCols = 2 * kBN;     // two accumulators
constexpr size_t kLmSmem = static_cast<size_t>(kStagesL) * kStageBytes + 1024;  // + alignment

// Instruction descriptor of tcgen05.mma kind::f16: float32 accumulator, bf16 A
// and B, both K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) |
                            ((kBM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand stored as 128-byte
// rows with the 128-byte swizzle: start address, stride between groups of
// eight rows (1024 bytes), descriptor version 1, swizzle mode 128 bytes.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr)
{
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;            // leading offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;    // stride offset
    d |= static_cast<uint64_t>(1u) << 46;            // version
    d |= static_cast<uint64_t>(2u) << 61;            // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 consecutive float32 columns of this thread's TMEM lane. The load and its
// wait sit in one asm statement, so no use of the registers can be scheduled
// between them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ bool finite_f(float x) { return fabsf(x) < __uint_as_float(0x7F800000u); }

// Which problem tile t belongs to, and its place there: vocabulary tile vt,
// row block rb (vocabulary-major, so the CTAs working at one time share a
// weight tile through L2).
struct TileAt {
    int p;
    int vt;
    int rb;
};

__device__ __forceinline__ TileAt tile_at(const LmArgs& a, int64_t t)
{
    const int p = (a.nprob > 1 && t >= a.p[0].tiles) ? 1 : 0;
    const int64_t lt = p ? t - a.p[0].tiles : t;
    const int nrb = a.p[p].n_rb;
    return TileAt{p, static_cast<int>(lt / nrb), static_cast<int>(lt % nrb)};
}

// Epilogue of one 128 x 256 tile for the 32 rows of this warp.
//  LOGITS: the float32 logits of the tile's valid columns to out[r * ldo + col].
//  STATS, sampling: one Partial per (row, vocabulary tile) -- the integer
//         reference exponent m = ceil(max x c) and the float-pair sum of
//         2^(x c - m) over the tile's columns -- and the draft token's raw
//         logit when the token falls in the tile.
//  STATS, greedy: the tile's largest raw logit and its lowest column.
// A NaN (or, when sampling, +inf) flags the row as non-finite.
template <int MODE>
__device__ __forceinline__ void epilogue_tile(const LmArgs& a, const TileAt& ti, uint32_t taddr,
                                              int q, int lane)
{
    const LmProblem& P = a.p[ti.p];
    const int64_t r = static_cast<int64_t>(ti.rb) * kBM + q * 32 + lane;
    const bool rv = r < P.R;
    const int64_t col_base = static_cast<int64_t>(ti.vt) * kBN;
    const int64_t ncols = a.V - col_base < kBN ? a.V - col_base : kBN;
    if (MODE == kLmLogits) {
        float* o = P.out + r * P.ldo + col_base;
        const bool vec = (P.ldo % 4 == 0) && ((reinterpret_cast<uintptr_t>(P.out) & 15) == 0);
        for (int ch = 0; ch < kBN / 32; ++ch) {
            float v[32];
            tmem_ld32(taddr + ch * 32, v);
            if (!rv) continue;
            if (vec && ch * 32 + 32 <= ncols) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(o + ch * 32 + j) =
                        make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (ch * 32 + j < ncols) o[ch * 32 + j] = v[j];
            }
        }
        return;
    }
    // The draft token this row verifies (row r = b per + i, i < K).
    int tcol = -1;
    if (rv && !a.greedy && P.per > 0) {
        const int64_t b = r / P.per, i = r - b * P.per;
        if (i < a.K) {
            const int64_t x = a.tokens[b * a.K + i];
            if (x >= col_base && x < col_base + ncols) tcol = static_cast<int>(x - col_base);
        }
    }
    const float ninf = __uint_as_float(kF32NegInfBits);
    float mx = ninf, tl = 0.f;
    int arg = INT_MAX, flags = 0;
    for (int ch = 0; ch < kBN / 32; ++ch) {
        float v[32];
        tmem_ld32(taddr + ch * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int col = ch * 32 + j;
            if (col < ncols) {
                const float x = v[j];
                if (x != x) flags = kFlagNonFinite;
                if (a.greedy) {
                    if (x > mx) {
                        mx = x;
                        arg = col;
                    }
                } else {
                    if (x == __uint_as_float(0x7F800000u)) flags = kFlagNonFinite;
                    mx = fmaxf(mx, x);
                }
            }
            if (col == tcol) tl = v[j];
        }
    }
    // Second read of the accumulator (sampling): the sum below the reference
    // exponent. Every lane of the warp takes part in each tcgen05.ld; rows
    // past the end and non-finite maxima only mask the terms.
    const float m = a.greedy ? mx : (finite_f(mx) ? ceilf(mx * a.c) : mx);
    float hi = 0.f, lo = 0.f;
    if (!a.greedy) {
        const bool fin = finite_f(m);
        const float nm = fin ? -m : 0.f;
        const int lim = fin ? static_cast<int>(ncols) : 0;
        for (int ch = 0; ch < kBN / 32; ++ch) {
            float v[32];
            tmem_ld32(taddr + ch * 32, v);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const int col = ch * 32 + j;
                s0 += col + 0 < lim ? ex2(fmaf(v[j + 0], a.c, nm)) : 0.f;
                s1 += col + 1 < lim ? ex2(fmaf(v[j + 1], a.c, nm)) : 0.f;
                s2 += col + 2 < lim ? ex2(fmaf(v[j + 2], a.c, nm)) : 0.f;
                s3 += col + 3 < lim ? ex2(fmaf(v[j + 3], a.c, nm)) : 0.f;
            }
            two_sum_acc(hi, lo, (s0 + s1) + (s2 + s3));
        }
    }
    if (!rv) return;
    Partial out;
    out.flags = flags;
    out.m = m;
    if (a.greedy) {
        out.hi = __int_as_float(arg == INT_MAX ? INT_MAX : static_cast<int>(col_base) + arg);
        out.lo = 0.f;
    } else {
        out.hi = hi;
        out.lo = lo;
        if (tcol >= 0) a.tok[P.row0 + r] = tl;
    }
    a.part[(P.row0 + r) * a.n_vt + ti.vt] = out;
}

// Wait for the last fill of every ring stage this thread issued (bounded), so
// that no bulk copy is still writing shared memory when the CTA exits after a
// wait ran out elsewhere.
__device__ __forceinline__ void drain_fills(uint64_t* full, int64_t issued)
{
    const int64_t first = issued > kStagesL ? issued - kStagesL : 0;
    for (int64_t j = first; j < issued; ++j)
        mbar_wait_bounded(&full[j % kStagesL], static_cast<uint32_t>((j / kStagesL) & 1), nullptr);
}

template <int MODE>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
                  const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1,
                  const __grid_constant__ LmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kStagesL], empty[kStagesL], tfull[2], tempty[2], done;
    __shared__ uint32_t tmem_base;
    __shared__ int stop;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_tiles = a.p[0].tiles + (a.nprob > 1 ? a.p[1].tiles : 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesL; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);  // one arrival per epilogue warp
        }
        mbar_init(&done, 1);
        stop = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    volatile int* vstop = &stop;
    auto fail = [&]() {
        *vstop = 1;
        atomicExch(a.err, 1);
    };

    if (warp == 0 && lane == 0) {
        // Producer: one k-block of both operands per ring stage.
        int64_t it = 0;
        bool ok = true;
        if (a.gate != nullptr) {
            // Test hook: hold every load until *gate != 0, with the same bound
            // as every other wait. Nothing sets it in the tests that use it, so
            // the wait runs out and the kernel takes its timeout path.
            const volatile int32_t* gate = a.gate;
            const long long t0 = clock64();
            while (*gate == 0) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    ok = false;
                    break;
                }
                __nanosleep(1000);
            }
        }
        for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            const TileAt ti = tile_at(a, t);
            const CUtensorMap* ma = ti.p ? &ta1 : &ta0;
            const CUtensorMap* mb = ti.p ? &tb1 : &tb0;
            const int nkb = a.p[ti.p].n_kb;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = static_cast<int>(it % kStagesL);
                const int64_t round = it / kStagesL;
                if (round > 0 &&
                    !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((round - 1) & 1), vstop)) {
                    ok = false;
                    break;
                }
                uint8_t* sa = base + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(sa, ma, kb * kBK, ti.rb * kBM, &full[s]);
                tma_load_2d(sa + kABytes, mb, kb * kBK, ti.vt * kBN, &full[s]);
            }
        }
        if (!ok) {
            fail();
            drain_fills(full, it);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: 128 x 256 x 16 per instruction, four per k-block.
        int64_t it = 0, tc = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tc) {
            const int acc = static_cast<int>(tc & 1);
            const int64_t use = tc >> 1;
            if (use > 0 &&
                !mbar_wait_bounded(&tempty[acc], static_cast<uint32_t>((use - 1) & 1), vstop)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(acc * kBN);
            const int nkb = a.p[tile_at(a, t).p].n_kb;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = static_cast<int>(it % kStagesL);
                const int64_t round = it / kStagesL;
                if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>(round & 1), vstop)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_addr(base + s * kStageBytes);
                const uint32_t sb = sa + kABytes;
#pragma unroll
                for (int k = 0; k < kBK / kUK; ++k)
                    mma_bf16(d, umma_desc(sa + k * kUK * 2), umma_desc(sb + k * kUK * 2),
                             (kb > 0 || k > 0) ? 1u : 0u);
                mma_commit(&empty[s]);  // the stage is free once these MMAs are done
            }
            if (!ok) break;
            mma_commit(&tfull[acc]);
        }
        if (!ok) fail();
        // Every MMA issued above has completed once this commit arrives.
        mma_commit(&done);
        mbar_wait_bounded(&done, 0, nullptr);
    } else if (warp >= 2) {
        // Epilogue: warp w reads TMEM lanes 32 (w mod 4) .. + 31.
        const int q = warp & 3;
        int64_t tc = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tc) {
            const int acc = static_cast<int>(tc & 1);
            const int64_t use = tc >> 1;
            const bool ok = mbar_wait_bounded(&tfull[acc], static_cast<uint32_t>(use & 1), vstop);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) fail();
                break;
            }
            tc_fence_after();
            const uint32_t taddr =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
            epilogue_tile<MODE>(a, tile_at(a, t), taddr, q, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// The hidden states of each sequence's emitted position j (from the scan's
// records), packed into [B, D] matrices: target row b (K + 1) + j and draft
// row b K + j (zeros for the bonus position j = K or an invalid sequence).
__global__ void gather_hidden_kernel(const uint8_t* ht, const uint8_t* hd, const SeqRecord* seqs,
                                     int64_t B, int64_t K, int64_t row_t, int64_t row_d,
                                     uint8_t* out_t, uint8_t* out_d)
{
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
    const SeqRecord rec = seqs[b];
    const int64_t j = rec.j;
    // (An emitted position outside [0, K] leaves zeros; the sampler, reading
    // the same record, reports the sequence.)
    const bool ok = rec.status == 0 && SV_IN_RANGE(j, K + 1);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < row_t / 16;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x)
        reinterpret_cast<uint4*>(out_t + b * row_t)[v] =
            ok ? reinterpret_cast<const uint4*>(ht + (b * (K + 1) + j) * row_t)[v] : z;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < row_d / 16;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x)
        reinterpret_cast<uint4*>(out_d + b * row_d)[v] =
            (ok && j < K) ? reinterpret_cast<const uint4*>(hd + (b * K + j) * row_d)[v] : z;
    }
}

// After a bounded wait in the LM head ran out: every sequence is reported as
// timed out (its tokens -1), whatever the later kernels wrote.
__global__ void lm_fail_kernel(const int32_t* err, int64_t B, int64_t K, int32_t* out_tokens,
                               int32_t* num_accepted, int32_t* seq_status)
{
    if (*err == 0) return;
    for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < B;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        for (int64_t i = 0; i <= K; ++i) out_tokens[b * (K + 1) + i] = -1;
        num_accepted[b] = -1;
        if (seq_status) seq_status[b] = kFlagTimeout;
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled lookup_encode()
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<EncodeTiled>(p);
    return nullptr;
}

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised once even when several host threads call at the same time).
EncodeTiled encode_fn()
{
    static const EncodeTiled fn = lookup_encode();
    return fn;
}

// A 2-D tensor map over a row-major bf16 matrix [rows, D], boxes of
// box_rows x 64 elements with the 128-byte swizzle; reads outside the matrix
// return zeros (ragged row blocks, vocabulary tiles and K).
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t D, int box_rows)
{
    EncodeTiled fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap* m, const LmArgs& a, int grid, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(lmhead_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kLmSmem));
    if (e != cudaSuccess) return e;
    lmhead_kernel<MODE><<<grid, kLmThreads, kLmSmem, s>>>(m[0], m[1], m[2], m[3], a);
    return cudaGetLastError();
}

}  // namespace

int64_t lmhead_vocab_tiles(int64_t V) { return (V + kBN - 1) / kBN; }

cudaError_t launch_lmhead(int mode, LmArgs a, cudaStream_t s, bool* mapped)
{
    CUtensorMap m[4];
    *mapped = true;
    for (int p = 0; p < a.nprob; ++p) {
        LmProblem& P = a.p[p];
        *mapped = *mapped && make_map(&m[2 * p], P.hidden, P.R, P.D, kBM) &&
                  make_map(&m[2 * p + 1], P.weights, a.V, P.D, kBN);
        P.n_rb = static_cast<int32_t>((P.R + kBM - 1) / kBM);
        P.n_kb = static_cast<int32_t>((P.D + kBK - 1) / kBK);
        P.tiles = static_cast<int64_t>(P.n_rb) * lmhead_vocab_tiles(a.V);
    }
    if (!*mapped) return cudaSuccess;
    if (a.nprob < 2) {
        m[2] = m[0];
        m[3] = m[1];
        a.p[1] = a.p[0];
        a.p[1].tiles = 0;
    }
    a.n_vt = static_cast<int32_t>(lmhead_vocab_tiles(a.V));
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int64_t tiles = a.p[0].tiles + (a.nprob > 1 ? a.p[1].tiles : 0);
    if (tiles == 0) return cudaSuccess;
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    return mode == kLmLogits ? launch_mode<kLmLogits>(m, a, grid, s)
                             : launch_mode<kLmStats>(m, a, grid, s);
}

cudaError_t launch_gather_hidden(const void* ht, const void* hd, const SeqRecord* seqs, int64_t B,
                                 int64_t K, int64_t Dt, int64_t Dd, void* out_t, void* out_d,
                                 cudaStream_t s)
{
    if (B == 0) return cudaSuccess;
    const dim3 grid(4, static_cast<unsigned>(B < 65535 ? B : 65535)), block(256);
    gather_hidden_kernel<<<grid, block, 0, s>>>(
        static_cast<const uint8_t*>(ht), static_cast<const uint8_t*>(hd), seqs, B, K, Dt * 2,
        Dd * 2, static_cast<uint8_t*>(out_t), static_cast<uint8_t*>(out_d));
    return cudaGetLastError();
}

cudaError_t launch_lm_fail(const int32_t* err, int64_t B, int64_t K, int32_t* out_tokens,
                           int32_t* num_accepted, int32_t* seq_status, cudaStream_t s)
{
    if (B == 0) return cudaSuccess;
    const int64_t blocks = (B + 255) / 256;
    lm_fail_kernel<<<static_cast<unsigned>(blocks < 1024 ? blocks : 1024), 256, 0, s>>>(
        err, B, K, out_tokens, num_accepted, seq_status);
    return cudaGetLastError();
}

}  // namespace sv
