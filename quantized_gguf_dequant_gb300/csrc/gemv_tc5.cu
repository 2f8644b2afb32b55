// gemv_tc5.cu -- batched decode of Q4_K (2..16 activation rows) on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// The operation: Y[t][n] = sum_k w[n][k] * X[t][k] for T <= 16 activation
// rows sharing one read of the weights -- the decode step of a server that
// batches requests ("Frink Inference: the Rust alternative to llama.cpp",
// "The goal, stated once": continuous batching), with the weights decoded
// inline ("Building a Rust Inference Engine That Matches Llama.cpp", "Where
// the wins came from").  fp32 activations, exact weights: every product is
// exact and the sums are fp32, as on the one-row path.
//
// Operands (fp16, kind::f16, fp32 accumulation):
//   A (the MMA's M side) = 256 weight rows x 64 k per step, each value
//     q * sc (a 4-bit code times its sub-block's 6-bit scale, at most 945:
//     exact in fp16), made by one fused fp16 multiply-add per two weights,
//     (1024 + q) * sc - 1024 * sc, from the nibble with 0x6400 above it;
//   B (the N side) = NC columns: token t's activations as two fp16 terms
//     hi + lo after an exact power-of-two scale 2^e per (token, super-block),
//     prepared once per call by tc5_prep_kernel.
// So D[n][2t] + D[n][2t+1] = 2^e * sum_k q sc x per super-block, and the
// epilogue adds d * 2^-e times that, minus dmin * sum_j m_j * (sum of x over
// sub-block j), for each row and token.  The k order inside each 64-wide step
// is the one that makes A cheapest: one 16-byte chunk of A holds the eight
// weights of one nibble word (bytes b0..b3) as (b0.lo, b2.lo), (b0.hi, b2.hi),
// (b1.lo, b3.lo), (b1.hi, b3.hi); the prep kernel writes x in the same order.
//
// Tiling: a work item is a 256-row tile x a slice of the super-blocks; K is
// cut into slices so that the items fill the SMs, each slice writes its
// partial sums, and the last slice of a tile to finish (a per-tile ticket)
// adds them in slice order -- bitwise repeatable.  Per 64-wide step two
// MMAs of M = 128 (the tile's halves) x N = NC x K = 16, four K steps; each
// super-block accumulates in its own tensor-memory buffer (two, alternating)
// so that the epilogue of one overlaps the MMAs of the next.
//
// Warp roles (576 threads, one CTA per SM):
//   warp 0      TMA producer: the rows' 16-byte headers once per super-block,
//               per step the rows' 32 nibble bytes and the B step (64 k x NC)
//   warp 1      tensor-memory allocation and MMA issue
//   warps 2..9  epilogue: tensor memory -> fp32, d / dmin / m_j scaling, sums
//   warps 10..17 A: one weight row per thread
// Every wait is bounded; a timeout raises the CTA's abort flag, the roles
// leave their loops, issued copies and MMAs are waited for, tensor memory is
// released.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "tcgen05.cuh"

namespace qmm {

namespace {

using namespace t5;

constexpr int kR = 256;               // weight rows per tile (two MMAs of M = 128)
constexpr int kABytes = kR * 128;     // fp16 A of one 64-wide step
constexpr int kNib = kR * 32;         // nibble bytes of one step
constexpr int kHdr = kR * 16;         // headers of one super-block
constexpr int kScl = 16 * 4;          // the super-block's 2^-e per token
constexpr int kXs = 128 * 4;          // its eight sub-block sums of x per token
// one header-ring slot; a multiple of 128 bytes, since a tensor copy's
// shared-memory destination must be 128-byte aligned
constexpr int kSlot = (kHdr + kScl + kXs + 127) / 128 * 128;
static_assert(kSlot % 128 == 0 && kHdr % 16 == 0 && kScl % 16 == 0, "slot alignment");
constexpr int kHdrSlots = 3;
constexpr int kStages = 4;
constexpr int kThreads = 576;
constexpr int kEpi0 = 2, kDeq0 = 10;

template <int NC>
struct Cfg {
    static constexpr int kBBytes = NC * 128;  // NC rows x 64 k of fp16
    static constexpr size_t kStageBytes = size_t(kABytes) + kBBytes + kNib;
    static constexpr uint32_t kTmemCols = 4 * NC;  // 2 buffers x 2 halves x NC
    static constexpr size_t kSmem = 1024 + kStages * kStageBytes + size_t(kHdrSlots) * kSlot + 256;
    // kind::f16: D f32 (bit 4), A and B f16 (0), both K-major, N/8 at 17, M/16 at 24
    static constexpr uint32_t kIdesc =
        (1u << 4) | (uint32_t(NC >> 3) << 17) | (uint32_t(128 >> 4) << 24);
    static_assert(kSmem <= 232448, "shared memory per block");
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
};

struct T5Params {
    CUtensorMap tm_hdr;  // weight bytes [N][row_bytes] u8, box 16 x 256
    CUtensorMap tm_nib;  // weight bytes, box 32 x 256
    CUtensorMap tm_b;    // prepared activations [NC][K] f16, box 64 x NC, 128-byte swizzle
    const float *scl;    // [NB][16]: 2^-e per (super-block, token)
    const float *xs;     // [NB][8][16]: sum of x over each sub-block, per token
    float *y;            // Y[t][n] at y + t * ldy + n
    int64_t ldy;
    float *ws;           // [S][tiles][256][16] slice partials (S > 1)
    unsigned *tickets;   // [tiles][8]: per tile and epilogue warp, zero between launches
    int N, T, NB, S, sbs, tiles, items;
    unsigned *status;
};

// One-dimensional bulk copy global -> shared (16-byte aligned, a multiple of
// 16 bytes), completing on bar.
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// f16x2 bits of (v, v) for a small integer v (exact in fp16).
__device__ __forceinline__ uint32_t h2_of(float v)
{
    const uint32_t h = __half_as_ushort(__float2half_rn(v));
    return h | (h << 16);
}

template <int NC>
__global__ void __launch_bounds__(kThreads, 1) gemv_tc5_kernel(const __grid_constant__ T5Params P)
{
    using C = Cfg<NC>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - smem_u32(smem_raw));
    // stage s: [A 32 KB][B NC x 128 B][nibbles 8 KB]
    auto sA = [&](int s) { return base + size_t(s) * C::kStageBytes; };
    auto sB = [&](int s) { return sA(s) + kABytes; };
    auto sNib = [&](int s) { return sB(s) + C::kBBytes; };
    uint8_t *sHdr = base + size_t(kStages) * C::kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sHdr + kHdrSlots * kSlot);
    uint64_t *full = bars;                  // nibbles + B landed        (tx)
    uint64_t *aready = full + kStages;      // A written                 (8 A warps)
    uint64_t *empty = aready + kStages;     // the step's MMAs done      (commit)
    uint64_t *hfull = empty + kStages;      // headers + scales + sums landed (tx)
    uint64_t *hempty = hfull + kHdrSlots;   // headers read              (8 A + 8 epilogue warps)
    uint64_t *accfull = hempty + kHdrSlots; // [2] super-block sums done (commit)
    uint64_t *accempty = accfull + 2;       // [2] sums read             (8 epilogue warps)
    uint64_t *drain = accempty + 2;         // final MMA drain           (commit)
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&aready[s], 8);
            mbar_init(&empty[s], 1);
        }
        for (int h = 0; h < kHdrSlots; ++h) {
            mbar_init(&hfull[h], 1);
            mbar_init(&hempty[h], 16);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], 8);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_sh)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    pdl_wait();  // the prepared activations (previous kernel) and Y

    auto item_of = [&](int it, int &tile, int &slice, int &sb0, int &sb1) {
        tile = it / P.S;
        slice = it - tile * P.S;
        sb0 = slice * P.sbs;
        sb1 = min(P.NB, sb0 + P.sbs);
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int st = 0, hit = 0;  // steps and headers issued
            bool ok = true;
            for (int it = blockIdx.x; it < P.items && ok; it += gridDim.x) {
                int tile, slice, sb0, sb1;
                item_of(it, tile, slice, sb0, sb1);
                const int row0 = tile * kR;
                for (int sb = sb0; sb < sb1 && ok; ++sb) {
                    const int h = hit % kHdrSlots, hu = hit / kHdrSlots;
                    if (hu >= 1 && !wait_phase(&hempty[h], unsigned(hu - 1) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *slot = sHdr + h * kSlot;
                    mbar_arrive_expect_tx(&hfull[h], kHdr + kScl + kXs);
                    tma_2d(slot, &P.tm_hdr, sb * 144, row0, &hfull[h]);
                    bulk_copy(slot + kHdr, P.scl + size_t(sb) * 16, kScl, &hfull[h]);
                    bulk_copy(slot + kHdr + kScl, P.xs + size_t(sb) * 128, kXs, &hfull[h]);
                    ++hit;
                    for (int c = 0; c < 4; ++c, ++st) {
                        const int s = st % kStages, u = st / kStages;
                        if (u >= 1 && !wait_phase(&empty[s], unsigned(u - 1) & 1u, &abort_flag, P.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], C::kBBytes + kNib);
                        tma_2d(sB(s), &P.tm_b, sb * 256 + c * 64, 0, &full[s]);
                        tma_2d(sNib(s), &P.tm_nib, sb * 144 + 16 + 32 * c, row0, &full[s]);
                    }
                }
            }
            // copies still in flight land before the CTA exits (bounded)
            for (int s = 0; s < kStages && s < st; ++s)
                mbar_wait_bounded(&full[s], unsigned((st - 1 - s) / kStages) & 1u, 200000000ll);
            for (int h = 0; h < kHdrSlots && h < hit; ++h)
                mbar_wait_bounded(&hfull[h], unsigned((hit - 1 - h) / kHdrSlots) & 1u, 200000000ll);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            int st = 0, g = 0;  // steps and super-blocks issued
            bool ok = true;
            for (int it = blockIdx.x; it < P.items && ok; it += gridDim.x) {
                int tile, slice, sb0, sb1;
                item_of(it, tile, slice, sb0, sb1);
                for (int sb = sb0; sb < sb1 && ok; ++sb, ++g) {
                    const int b = g & 1, u = g >> 1;
                    if (u >= 1 && !wait_phase(&accempty[b], unsigned(u - 1) & 1u, &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int c = 0; c < 4; ++c, ++st) {
                        const int s = st % kStages, us = st / kStages;
                        if (!wait_phase(&full[s], unsigned(us) & 1u, &abort_flag, P.status) ||
                            !wait_phase(&aready[s], unsigned(us) & 1u, &abort_flag, P.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(sA(s)), b0 = smem_u32(sB(s));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t bd = sw128_desc(b0 + 32 * kk);
                            const uint32_t acc = (c | kk) != 0 ? 1u : 0u;
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                mma_f16(tmem + uint32_t((2 * b + h) * NC),
                                        sw128_desc(a0 + h * 16384 + 32 * kk), bd, C::kIdesc, acc);
                        }
                        mma_commit(&empty[s]);
                    }
                    if (!ok)
                        break;
                    mma_commit(&accfull[b]);
                }
            }
            mma_commit(drain);  // every MMA issued has finished once this arrives
            mbar_wait_bounded(drain, 0u, 200000000ll);
        }
    } else if (warp < kDeq0) {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp & 3;                // tensor-memory lanes 32*quarter ..
        const int half = (warp - kEpi0) >> 2;        // rows 128*half ..
        const int r = half * 128 + quarter * 32 + lane;  // weight row within the tile
        const uint32_t lane_base = uint32_t(quarter * 32) << 16;
        int g = 0, hit = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < P.items && ok; it += gridDim.x) {
            int tile, slice, sb0, sb1;
            item_of(it, tile, slice, sb0, sb1);
            float acc[16];
#pragma unroll
            for (int t = 0; t < 16; ++t)
                acc[t] = 0.f;
            for (int sb = sb0; sb < sb1; ++sb, ++g, ++hit) {
                const int b = g & 1, u = g >> 1;
                const int h = hit % kHdrSlots;
                if (!wait_phase(&accfull[b], unsigned(u) & 1u, &abort_flag, P.status) ||
                    !wait_phase(&hfull[h], unsigned(hit / kHdrSlots) & 1u, &abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t D[NC];
                const uint32_t taddr = tmem + lane_base + uint32_t((2 * b + half) * NC);
                tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(D));
                if constexpr (NC == 32)
                    tmem_ld16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(D + 16));
                tmem_ld_wait();
                const uint8_t *slot = sHdr + h * kSlot;
                const uint4 hd = *reinterpret_cast<const uint4 *>(slot + r * 16);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&accempty[b]);  // this buffer may take the next sums
                const float2 dd = half2_bits_to_float2(hd.x);  // (d, dmin)
                const float *scl = reinterpret_cast<const float *>(slot + kHdr);
                const float *xs = reinterpret_cast<const float *>(slot + kHdr + kScl);
                // min term: sum_j m_j * (sum of x over sub-block j), tokens in pairs
                float2 mn[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    mn[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t sc_, m_;
                    scale_min(hd.y, hd.z, hd.w, j, sc_, m_);
                    const float2 mj = make_float2(float(m_), float(m_));
                    const float4 *xj = reinterpret_cast<const float4 *>(xs + 16 * j);
#pragma unroll
                    for (int q = 0; q < NC / 8; ++q) {  // tokens 4q .. 4q+3
                        const float4 v = xj[q];
                        mn[2 * q] = __ffma2_rn(mj, make_float2(v.x, v.y), mn[2 * q]);
                        mn[2 * q + 1] = __ffma2_rn(mj, make_float2(v.z, v.w), mn[2 * q + 1]);
                    }
                }
#pragma unroll
                for (int q = 0; q < NC / 8; ++q) {
                    const float4 s4 = reinterpret_cast<const float4 *>(scl)[q];
                    const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = 4 * q + i;
                        const float main_t = __uint_as_float(D[2 * t]) + __uint_as_float(D[2 * t + 1]);
                        const float mn_t = (i & 1) ? mn[t >> 1].y : mn[t >> 1].x;
                        acc[t] = fmaf(dd.x * sv[i], main_t, acc[t]);
                        acc[t] = fmaf(-dd.y, mn_t, acc[t]);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&hempty[h]);  // the slot's scales and sums are read
            }
            if (!ok)
                break;
            // ---- the item's rows: out, or slice partials + the ordered sum
            const int row = tile * kR + r;
            if (P.S == 1) {
                if (row < P.N) {
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (t < P.T)
                            P.y[int64_t(t) * P.ldy + row] = acc[t];
                }
            } else {
                // Each epilogue warp owns its 32 rows end to end: it writes
                // their slice partials, takes the (tile, warp) ticket, and the
                // warp that completes the set adds the slices in slice order.
                float4 *wp = reinterpret_cast<float4 *>(
                    P.ws + ((size_t(slice) * P.tiles + tile) * kR + r) * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    wp[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                __threadfence();
                __syncwarp();
                unsigned last = 0;
                if (lane == 0) {
                    unsigned *tk = P.tickets + size_t(tile) * 8 + (warp - kEpi0);
                    last = atomicAdd(tk, 1u) == unsigned(P.S - 1) ? 1u : 0u;
                    if (last)
                        *tk = 0u;  // for the next launch
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    float sum[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        sum[t] = 0.f;
                    for (int sl = 0; sl < P.S; ++sl) {
                        const float4 *rp = reinterpret_cast<const float4 *>(
                            P.ws + ((size_t(sl) * P.tiles + tile) * kR + r) * 16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 v = __ldcg(rp + q);
                            sum[4 * q] += v.x;
                            sum[4 * q + 1] += v.y;
                            sum[4 * q + 2] += v.z;
                            sum[4 * q + 3] += v.w;
                        }
                    }
                    if (row < P.N) {
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            if (t < P.T)
                                P.y[int64_t(t) * P.ldy + row] = sum[t];
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------------- A (q * sc, fp16)
        const int r = (warp - kDeq0) * 32 + lane;  // weight row within the tile
        const uint32_t swz = uint32_t(r & 7);
        const uint32_t magic = 0x64006400u;  // 1024 in both halves
        int st = 0, hit = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < P.items && ok; it += gridDim.x) {
            int tile, slice, sb0, sb1;
            item_of(it, tile, slice, sb0, sb1);
            for (int sb = sb0; sb < sb1 && ok; ++sb, ++hit) {
                const int h = hit % kHdrSlots;
                if (!wait_phase(&hfull[h], unsigned(hit / kHdrSlots) & 1u, &abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                const uint4 hd = *reinterpret_cast<const uint4 *>(sHdr + h * kSlot + r * 16);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&hempty[h]);
                for (int c = 0; c < 4; ++c, ++st) {
                    const int s = st % kStages, u = st / kStages;
                    if (!wait_phase(&full[s], unsigned(u) & 1u, &abort_flag, P.status) ||
                        (u >= 1 && !wait_phase(&empty[s], unsigned(u - 1) & 1u, &abort_flag, P.status))) {
                        ok = false;
                        break;
                    }
                    uint32_t sc_lo, m_lo, sc_hi, m_hi;
                    scale_min(hd.y, hd.z, hd.w, 2 * c, sc_lo, m_lo);
                    scale_min(hd.y, hd.z, hd.w, 2 * c + 1, sc_hi, m_hi);
                    const uint32_t slo = h2_of(float(sc_lo)), shi = h2_of(float(sc_hi));
                    const uint32_t olo = h2_of(-1024.f * float(sc_lo)), ohi = h2_of(-1024.f * float(sc_hi));
                    const uint8_t *nib = sNib(s) + r * 32;
                    const uint4 n0 = *reinterpret_cast<const uint4 *>(nib);
                    const uint4 n1 = *reinterpret_cast<const uint4 *>(nib + 16);
                    const uint32_t w[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
                    uint8_t *arow = sA(s) + r * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t v = w[j];
                        const uint32_t p0 = hfma2_bits((v & 0x000F000Fu) | magic, slo, olo);
                        const uint32_t p1 = hfma2_bits(((v >> 4) & 0x000F000Fu) | magic, shi, ohi);
                        const uint32_t p2 = hfma2_bits(((v >> 8) & 0x000F000Fu) | magic, slo, olo);
                        const uint32_t p3 = hfma2_bits(((v >> 12) & 0x000F000Fu) | magic, shi, ohi);
                        *reinterpret_cast<uint4 *>(arow + ((uint32_t(j) ^ swz) << 4)) =
                            make_uint4(p0, p1, p2, p3);
                    }
                    fence_proxy_async_smem();  // the MMA reads A through the async proxy
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&aready[s]);
                }
            }
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ activations

// One warp per (token, super-block): the power-of-two scale that puts the
// super-block's largest |x| in [2^14, 2^15), the hi / lo fp16 terms in the
// A chunks' k order, and the eight sub-block sums of x.  Tokens t >= T (up
// to NC / 2) get zero columns.
__global__ void __launch_bounds__(256) tc5_prep_kernel(const float *__restrict__ X, int64_t ldx,
                                                       int T, int NB, int ncols, __half *Bg,
                                                       float *scl, float *xs)
{
    pdl_wait();  // X may come from the previous kernel
    pdl_launch_dependents();
    const int wid = int(blockIdx.x) * 8 + int(threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int t = wid / NB, sb = wid - t * NB;
    if (t >= ncols / 2)
        return;
    const int64_t K = int64_t(NB) * 256;
    float v[8];
    if (t < T) {
        const float4 *src = reinterpret_cast<const float4 *>(X + int64_t(t) * ldx + int64_t(sb) * 256) + 2 * lane;
        const float4 a = __ldg(src), b = __ldg(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = 0.f;
    }
    float mx = 0.f, s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        mx = fmaxf(mx, fabsf(v[i]));
        s += v[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // sub-block j = values 32j .. 32j+31 = lanes 4j .. 4j+3
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    int e = 0;
    if (mx > 0.f) {
        int E;
        frexpf(mx, &E);  // mx = f * 2^E, f in [0.5, 1)
        e = min(15 - E, 126);
    }
    if (lane == 0)
        scl[size_t(sb) * 16 + t] = scale_pow2(1.f, -e);
    if ((lane & 3) == 0)
        xs[size_t(sb) * 128 + (lane >> 2) * 16 + t] = s;
    __half *hi_row = Bg + size_t(2 * t) * K + int64_t(sb) * 256;
    __half *lo_row = Bg + size_t(2 * t + 1) * K + int64_t(sb) * 256;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int k = 8 * lane + i;  // natural position within the super-block
        const int c = k >> 6, kn = k & 63;
        const int beta = kn & 31, hiN = kn >> 5;  // nibble byte, high nibble?
        const int j = beta >> 2, bi = beta & 3;
        // position within the chunk: (b0.lo, b2.lo, b0.hi, b2.hi, b1.lo, b3.lo, b1.hi, b3.hi)
        const int p = ((bi & 1) << 2) | (hiN << 1) | (bi >> 1);
        const int pos = 64 * c + 8 * j + p;
        const float xv = scale_pow2(v[i], e);
        const __half hv = __float2half_rn(xv);
        const __half lv = __float2half_rn(xv - __half2float(hv));
        hi_row[pos] = hv;
        lo_row[pos] = lv;
    }
}

} // namespace

// ------------------------------------------------------------------ host

Tc5Plan plan_tc5(int64_t N, int64_t K, int T, int sm_count)
{
    Tc5Plan p;
    p.nc = T <= 8 ? 16 : 32;
    p.tiles = int((N + kR - 1) / kR);
    const int NB = int(K / 256);
    double best = 1e30;
    for (int S = 1; S <= std::min(NB, 16); ++S) {
        const int sbs = (NB + S - 1) / S;
        const int s_eff = (NB + sbs - 1) / sbs;
        if (s_eff != S)
            continue;
        const int64_t items = int64_t(p.tiles) * S;
        const double waves = double((items + sm_count - 1) / sm_count);
        const double t = waves * sbs + (S > 1 ? 0.5 : 0.0);
        if (t < best - 1e-9) {
            best = t;
            p.S = S;
            p.sbs = sbs;
        }
    }
    if (const char *e = getenv("QMM_TC5_S")) {  // a fixed slice count (tests, tuning)
        const int f = atoi(e);
        if (f >= 1 && f <= std::min(NB, 16)) {
            p.sbs = (NB + f - 1) / f;
            p.S = (NB + p.sbs - 1) / p.sbs;
        }
    }
    p.items = p.tiles * p.S;
    p.smem = p.nc == 16 ? Cfg<16>::kSmem : Cfg<32>::kSmem;
    p.ws_floats = p.S > 1 ? size_t(p.S) * p.tiles * kR * 16 : 0;
    p.tickets = size_t(p.tiles) * 8;
    p.prep_bytes = size_t(p.nc) * size_t(K) * 2 + size_t(NB) * 16 * 4 + size_t(NB) * 128 * 4;
    return p;
}

cudaError_t launch_gemv_tc5(const Tc5Plan &p, const Tc5Args &a, int sm_count, cudaStream_t s)
{
    const int NB = int(a.K / 256);
    __half *Bg = reinterpret_cast<__half *>(a.prep);
    float *scl = reinterpret_cast<float *>(static_cast<uint8_t *>(a.prep) + size_t(p.nc) * a.K * 2);
    float *xs = scl + size_t(NB) * 16;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cfg.stream = s;
    const int warps = (p.nc / 2) * NB;
    cfg.gridDim = dim3(unsigned((warps + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cudaError_t e = counted(cudaLaunchKernelEx(&cfg, tc5_prep_kernel, a.X, a.ldx, a.T, NB, p.nc,
                                               Bg, scl, xs));
    if (e != cudaSuccess)
        return e;
    T5Params P;
    memset(&P, 0, sizeof(P));
    memcpy(&P.tm_hdr, a.tmap_hdr, sizeof(CUtensorMap));
    memcpy(&P.tm_nib, a.tmap_nib, sizeof(CUtensorMap));
    memcpy(&P.tm_b, a.tmap_b, sizeof(CUtensorMap));
    P.scl = scl;
    P.xs = xs;
    P.y = a.Y;
    P.ldy = a.ldy;
    P.ws = a.ws;
    P.tickets = a.tickets;
    P.N = int(a.N);
    P.T = a.T;
    P.NB = NB;
    P.S = p.S;
    P.sbs = p.sbs;
    P.tiles = p.tiles;
    P.items = p.items;
    P.status = a.status;
    auto kern = p.nc == 16 ? gemv_tc5_kernel<16> : gemv_tc5_kernel<32>;
    e = func_smem(reinterpret_cast<const void *>(kern), p.smem);
    if (e != cudaSuccess)
        return e;
    cfg.gridDim = dim3(unsigned(std::min(p.items, sm_count)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    return counted(cudaLaunchKernelEx(&cfg, kern, P));
}

} // namespace qmm
