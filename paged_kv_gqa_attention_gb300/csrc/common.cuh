// Device helpers shared by the attention kernels: bf16 packing, the base-2
// exponential, warp reductions, mbarriers, bulk async copies and bounded
// waits.  Everything here is sm_103a-only inline PTX or plain CUDA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qa.h"

namespace qa {

// Bounded waits give up after this many nanoseconds (globaltimer), set
// QA_DEVICE_TIMEOUT and let the kernel run to its end instead of hanging.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// log2(e): scores are kept pre-multiplied by it so that exp(x) = 2^(x*log2e).
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32); 2^-inf = 0.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 pair in one 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> packed bf16 pair, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Packed fp32 pairs (sm_100 family f32x2 instructions): one instruction
// operates on both halves of a 64-bit register pair.
__device__ __forceinline__ uint64_t f2_bits(float2 a) { return *reinterpret_cast<uint64_t *>(&a); }
__device__ __forceinline__ float2 bits_f2(uint64_t b) { return *reinterpret_cast<float2 *>(&b); }

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// cos/sin of pos * f for an integer position 0 <= pos < 2^18 and a frequency
// f = f_hi + f_lo (f_hi = f rounded to fp32, f_lo the fp32 rounding of the
// rest), in fp32 without fp64 arithmetic: the product is carried as
// a_hi + a_lo + pos * f_lo (a_lo the exact FMA residual of pos * f_hi), and
// reduced modulo 2 pi by the three-constant Cody-Waite scheme (W. J. Cody and
// W. Waite, "Software Manual for the Elementary Functions", 1980): 2 pi =
// C1 + C2 + C3 with C1 = 6.28125 (8 significant bits), so n * C1 is exact for
// n < 2^16 and the first subtraction is exact.  The reduced angle is within a
// few fp32 ulps of the true one, then an fp32 sincos.
__device__ __forceinline__ void sincos_pos_freq(int pos, float f_hi, float f_lo, float *s, float *c) {
    constexpr double kTwoPiD = 6.283185307179586476925286766559;
    constexpr float kC1 = 6.28125f;
    constexpr float kC2 = (float)(kTwoPiD - 6.28125);
    constexpr float kC3 = (float)(kTwoPiD - 6.28125 - (double)(float)(kTwoPiD - 6.28125));
    constexpr float kInvTwoPi = (float)(1.0 / kTwoPiD);
    const float p = (float)pos;
    const float a_hi = p * f_hi;
    const float a_lo = fmaf(p, f_hi, -a_hi) + p * f_lo;
    const float n = rintf(a_hi * kInvTwoPi);
    float r = fmaf(-n, kC1, a_hi);
    r = fmaf(-n, kC2, r);
    r = fmaf(-n, kC3, r);
    sincosf(r + a_lo, s, c);
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns (kWaitLimitNs unless a check passes a shorter one), ORs
// QA_DEVICE_TIMEOUT into *status and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int *status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, QA_DEVICE_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------- bulk copies
// One contiguous global -> shared copy completed on an mbarrier (the bulk
// copy engine, no tensor map).  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same with an L2 eviction-priority hint (createpolicy evict_first): data
// streamed exactly once should not push reusable lines out of L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Named barrier over `count` threads (a multiple of 32); id 0 is __syncthreads.
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace qa
