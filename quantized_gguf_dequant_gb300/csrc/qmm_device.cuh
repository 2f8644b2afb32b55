// qmm_device.cuh -- device-side building blocks shared by the kernels:
// mbarrier + bulk-copy (TMA engine) staging, programmatic dependent launch,
// bounded waits that report through the handle's status word, and the small
// bit-level helpers of the Q4_K / Q8_0 decoders.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace qmm {

// A pipeline wait gives up after this many SM clock cycles (about a second at
// GB300 clocks): far beyond any legitimate wait, short enough that a broken
// pipeline returns an error instead of hanging the GPU.
constexpr long long kWaitBudgetCycles = 2000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe: has phase `parity` of the mbarrier completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread may sleep (up to the hint,
// in ns) until the phase completes instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after `budget` cycles.
// Returns false on timeout (the caller records it and winds down).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity,
                                                  long long budget = kWaitBudgetCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_sleep(bar, parity))
                return true;
        if (clock64() - t0 > budget)
            return false;
    }
}

// ----------------------------------------------------------------- bulk copy
// Fetch a TMA descriptor (a kernel parameter's generic address) into the
// descriptor cache ahead of its first copy, e.g. while the previous kernel in
// the stream drains.
__device__ __forceinline__ void prefetch_tmap(const void *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// One-dimensional bulk copy global -> shared through the TMA engine,
// completing `bytes` transactions on `bar`.  dst, src 16-byte aligned, bytes a
// multiple of 16.  The L2 policy marks the (read-once) weight stream
// evict-first so it does not push reusable data out of L2.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes,
                                         uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ----------------------------------------------------------------- PDL
// Programmatic dependent launch: the next kernel in the stream may start its
// prologue (constant-weight prefetch) once every CTA of this one has called
// launch_dependents; it must call wait before touching anything this kernel
// writes (outputs, workspace) or anything an earlier kernel produced (inputs).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- bits
__device__ __forceinline__ float as_float(uint32_t u) { return __uint_as_float(u); }

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }

// x * 2^e exactly (two power-of-two factors so that e may span [-252, 254]),
// unless the result itself over- or underflows.
__device__ __forceinline__ float scale_pow2(float x, int e)
{
    const int e1 = e / 2;
    return (x * exp2i(e1)) * exp2i(e - e1);
}

// The float 2^23 + b for a byte b taken from position k (0..3) of v:
// bytes [v.b_k, 0, 0, 0x4B].  Subtracting 2^23 afterwards gives b exactly.
__device__ __forceinline__ float byte_magic(uint32_t v, int k)
{
    return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7540u | unsigned(k)));
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h)
{
    return make_float2(__half2float(__ushort_as_half((unsigned short)(h & 0xffffu))),
                       __half2float(__ushort_as_half((unsigned short)(h >> 16))));
}

__device__ __forceinline__ float warp_sum(float v, int width)
{
    for (int o = width >> 1; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

} // namespace qmm
