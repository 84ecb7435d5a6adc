// PTX wrappers shared by the state kernels (sm_103a): mbarriers, bulk copies
// from global to shared memory, packed fp32 arithmetic.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Every mbarrier wait is bounded in time: it gives up kWaitNs after it began
// (the %globaltimer clock, nanoseconds), and in any case after kWaitRounds
// suspended try_wait rounds.  A round suspends for at most about the hint when
// the barrier is idle, but can take much longer; the clock is the bound that
// holds in practice.
constexpr unsigned long long kWaitNs = 1000000000ull; // 1 s
constexpr long long kWaitRounds = 1ll << 26;
constexpr uint32_t kSuspendHintNs = 1000;

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t sm_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// try_wait suspends the thread until the phase completes or the hint (ns)
// runs out, so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
                 : "memory");
    return ok != 0;
}
// Bounded wait for the phase of `parity` to complete; false when it ran out
// (after `limit_ns` nanoseconds, or kWaitRounds rounds).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns = kWaitNs)
{
    if (mbar_try(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (long long i = 0; i < kWaitRounds; ++i) {
        if (mbar_try(bar, parity))
            return true;
        if (global_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// Two-wide fp32 FMA and multiply: each half rounds exactly like the scalar op.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    unsigned long long A = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long B = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long Cc = *reinterpret_cast<unsigned long long *>(&c);
    unsigned long long D;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(A), "l"(B), "l"(Cc));
    return *reinterpret_cast<float2 *>(&D);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    unsigned long long A = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long B = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long D;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(D) : "l"(A), "l"(B));
    return *reinterpret_cast<float2 *>(&D);
}

} // namespace gdn
