// tcgen05.cuh -- PTX wrappers of the 5th-generation tensor-core paths (the
// prefill GEMM and the batched decode): 2-D TMA loads, the 128-byte-swizzle
// K-major shared-memory descriptor, MMA commits, tensor-memory loads and
// fences, and bounded pipeline waits that raise a CTA-wide abort flag.
#pragma once

#include <cstdint>

#include <cuda.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace t5 {

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y,
                                       uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Tiled bulk stores shared -> global (one tensor-map box), in the calling
// thread's bulk group; rows or columns past the tensor's extent are not
// written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
                 "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core
// groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t(1) << 16;            // leading byte offset (unused for this layout)
    d |= uint64_t(1024 >> 4) << 32;    // stride byte offset
    d |= uint64_t(1) << 46;            // version
    d |= uint64_t(2) << 61;            // 128-byte swizzle
    return d;
}

// The mbarrier completes one arrival when every tcgen05 operation this
// thread issued so far has finished.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Bounded wait that also gives up when another role raised the abort flag.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, unsigned parity, volatile int *abort,
                                           unsigned *status)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_sleep(bar, parity))
                return true;
        if (*abort)
            return false;
        if (clock64() - t0 > kWaitBudgetCycles) {
            atomicOr(status, kStatusTimeoutBit);
            *abort = 1;
            return false;
        }
    }
}

// The (sc, m) pair of sub-block j (0..7) from the 12 packed scale bytes
// q[0..11] held in words s0 = q[0..3], s1 = q[4..7], s2 = q[8..11].
__device__ __forceinline__ void scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j,
                                          uint32_t &sc, uint32_t &m)
{
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63u;
        m = (s1 >> (8 * j)) & 63u;
    } else {
        const int i = j - 4;
        const uint32_t b = (s2 >> (8 * i)) & 0xFFu;
        sc = (b & 0x0Fu) | (((s0 >> (8 * i + 6)) & 3u) << 4);
        m = (b >> 4) | (((s1 >> (8 * i + 6)) & 3u) << 4);
    }
}

// tcgen05.mma kind::f16 (fp32 accumulate in tensor memory); idesc carries
// the operand types and the M x N shape.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

} // namespace t5
} // namespace qmm
