// sv_device.cuh -- device helpers for the verification kernels (sm_103a).
//
// Inline PTX for the pieces CUDA C++ does not expose directly: mbarrier
// waits with a time limit, 1-D bulk copies global -> shared (the TMA engine's
// untiled form), the SFU base-2 exponential, and NaN-propagating maxima on
// packed bfloat16 pairs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// ---------------------------------------------------------------------------
// Device-side index checks
// ---------------------------------------------------------------------------
// Built with -DSV_DEVICE_CHECKS (the library's debug variant), SV_IN_RANGE(i,
// n) tests 0 <= i < n where a kernel indexes memory by a value it computed or
// read; a kernel whose test fails skips that access and reports kFlagIndex
// (SV_SEQ_INDEX) for the row or sequence it was working on, never a trap.
// In the product build the tests are the constant true and cost nothing.
#ifdef SV_DEVICE_CHECKS
constexpr bool kDeviceChecks = true;
#define SV_IN_RANGE(i, n) \
    (static_cast<long long>(i) >= 0 && static_cast<long long>(i) < static_cast<long long>(n))
#else
constexpr bool kDeviceChecks = false;
#define SV_IN_RANGE(i, n) true
#endif

// ---------------------------------------------------------------------------
// Arithmetic
// ---------------------------------------------------------------------------
// 2^x on the special-function unit (ex2.approx, subnormal results flushed).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max with NaN propagation: the result is NaN if either input is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Lane-wise max of two packed bfloat16 pairs, NaN-propagating.
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The two bfloat16 halves of a 32-bit word, widened exactly to float.
// Element 2w sits in the low half (little-endian), element 2w+1 in the high.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

constexpr uint32_t kBf16NegInfPair = 0xFF80FF80u;
constexpr uint32_t kF32NegInfBits = 0xFF800000u;

// 2^d for an integer-valued float d <= 0 (or -inf), built exactly from bits;
// 0 below the normal range.
__device__ __forceinline__ float pow2_neg_int(float d)
{
    if (!(d > -126.0f)) return 0.0f;
    return __int_as_float((127 + static_cast<int>(d)) << 23);
}

// hi + lo += x with the rounding error of the high sum kept in lo (Knuth's
// two-sum; no assumption on the magnitudes).
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float x)
{
    const float s = __fadd_rn(hi, x);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
    hi = s;
    lo = __fadd_rn(lo, err);
}

// Knuth's two-sum: s + err == a + b exactly (round to nearest, no overflow).
__device__ __forceinline__ float two_sum(float a, float b, float* err)
{
    const float s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    *err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
    return s;
}

// (hi + lo) * 2^m  +=  (ohi + olo) * 2^om, both exponents integer-valued or
// -inf (an empty sum). The rescales are exact powers of two, so the only
// rounding is the one two-sum keeps in lo.
__device__ __forceinline__ void merge_scaled(float& m, float& hi, float& lo, float om, float ohi,
                                             float olo)
{
    const float M = fmaxf(m, om);
    if (M == __uint_as_float(0xFF800000u)) return;  // both empty
    const float a = pow2_neg_int(m - M), b = pow2_neg_int(om - M);
    float err;
    const float s = two_sum(__fmul_rn(hi, a), __fmul_rn(ohi, b), &err);
    lo = __fadd_rn(__fadd_rn(__fmul_rn(lo, a), __fmul_rn(olo, b)), err);
    hi = s;
    m = M;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11, section 4). Ten rounds of
// two 32x32 multiplies (words 0 and 2) whose high halves are xored with the
// other words and the round key; the key advances by the two Weyl increments.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint2 k)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t a = x.x, c = x.z;
        const uint32_t lo_a = a * 0xD2511F53u, hi_a = __umulhi(a, 0xD2511F53u);
        const uint32_t lo_c = c * 0xCD9E8D57u, hi_c = __umulhi(c, 0xCD9E8D57u);
        x = make_uint4(hi_c ^ x.y ^ k.x, lo_c, hi_a ^ x.w ^ k.y, lo_a);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return x;
}

// The verifier's uniforms: counter (pos, seq, 0, 0), key = (lo, hi) of seed.
__device__ __forceinline__ uint4 verify_random_words(uint64_t seed, uint32_t seq, uint32_t pos)
{
    return philox4x32_10(make_uint4(pos, seq, 0u, 0u),
                         make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)));
}
// 24-bit uniform in [0, 1 - 2^-24]; exact in float.
__device__ __forceinline__ float word_to_uniform(uint32_t w)
{
    return static_cast<float>(w >> 8) * 5.9604644775390625e-8f;
}
// Race uniform in (0, 1): (2 (w >> 9) + 1) * 2^-24, exact in float.
__device__ __forceinline__ float word_to_open_uniform(uint32_t w)
{
    return static_cast<float>(2u * (w >> 9) + 1u) * 5.9604644775390625e-8f;
}
// -ln v for v in (0, 1) with full relative precision near v = 1.
__device__ __forceinline__ float exp_clock(float v) { return -log1pf(v - 1.0f); }

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream is still
// running; pdl_wait() blocks until that kernel has completed and its memory
// is visible (and returns at once when the kernel was launched normally).
// pdl_trigger() lets the next kernel start launching once every CTA of this
// one has issued it or exited.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory mbarriers and bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// One wait for phase `parity` of `bar`: the thread may be suspended until the
// phase completes or about `suspend_ns` nanoseconds have passed (a hint; the
// hardware wakes the thread when the phase completes, so waiting warps spend
// no issue slots). True if the phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t suspend_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// Upper bound on any wait inside the kernels, in SM clock cycles (about two
// seconds at 2 GHz). A wait that runs out returns false; the caller records a
// timeout status and winds down instead of spinning forever.
constexpr long long kWaitLimitCycles = 4000000000LL;
// Suspend hint of one try: 1 ms, so the time limit is checked often enough.
constexpr uint32_t kSuspendHintNs = 1000000u;

// Wait for phase `parity` of `bar`. Gives up when *abort becomes non-zero
// (another thread of the CTA already gave up) or after kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const volatile int* abort)
{
    if (mbar_try_wait(bar, parity, kSuspendHintNs)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity, kSuspendHintNs)) return true;
        if (abort != nullptr && *abort != 0) return false;
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Read-only scalar loads of one logit, widened to float.
__device__ __forceinline__ float load_logit_bf16(const void* p)
{
    const uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ float load_logit_f32(const void* p)
{
    return __ldg(reinterpret_cast<const float*>(p));
}

}  // namespace sv
