// tc_common.cuh -- building blocks of the tensor-core Q4_K kernels (decode
// GEMV and the expert GEMV): the fp16 operand construction from packed
// nibbles, the super-block header decode, the activation -> B-fragment
// layout, mma.sync and 2-D TMA wrappers, and the per-unit dot product.
// The layout conventions are described at the top of gemv_tc.cu.
#pragma once

#include <cuda.h>

#include "qmm_device.cuh"

namespace qmm {
namespace tc {

constexpr int kTileRows = 16;
constexpr int kTileBytes = kTileRows * 144;  // 2304

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (a & b) | c in one LOP3 (lookup table 0xEA); written out because the
// compiler otherwise splits a mask-and-merge with two constants in two.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// D = A B (+ C) with fp16 operands and fp32 accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    const float z = 0.f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Per-row decode of the super-block header for chunk c: the fp16 pairs the
// operand construction needs, and (d, dmin).
struct RowScales {
    uint32_t SL, CL, SH, CH;  // (sc_lo, sc_lo), -1024*SL, (sc_hi/16, ..), -1024*SH
    uint32_t Am;              // (m_lo, m_hi)
    float d, dmin;
};

__device__ __forceinline__ RowScales row_scales(uint4 h, uint32_t selA, uint32_t selB, bool hi4)
{
    const uint32_t A = __byte_perm(h.y, h.z, selA);
    const uint32_t B = __byte_perm(h.w, h.w, selB);
    const uint32_t R = hi4 ? (((B & 0x00000F0Fu) | ((B >> 4) & 0x0F0F0000u)) |
                              ((A >> 2) & 0x30303030u))
                           : (A & 0x3F3F3F3Fu);  // bytes: sc_lo, sc_hi, m_lo, m_hi
    RowScales s;
    // 0x64vv is the fp16 1024 + v; subtracting 1024 (0xE400) leaves v exactly.
    s.SL = hadd2(__byte_perm(R, 0x64u, 0x4040u), 0xE400E400u);
    s.SH = hfma2(__byte_perm(R, 0x64u, 0x4141u), 0x2C002C00u, 0xD400D400u);  // (1024+v)/16 - 64
    s.CL = hmul2(s.SL, 0xE400E400u);
    s.CH = hmul2(s.SH, 0xE400E400u);
    s.Am = hadd2(__byte_perm(R, 0x64u, 0x4342u), 0xE400E400u);
    const float2 dd = half2_bits_to_float2(h.x);
    s.d = dd.x;
    s.dmin = dd.y;
    return s;
}

// Activations of super-block sb, x row m, as this lane's share of the B
// fragments (see the fragment layout above), the sub-block sums for the min
// MMA, and the inverse scale.  Lane (cc, tt) = (lane >> 3, lane & 7) holds
// x[64cc + 4tt .. +3] (v) and x[64cc + 32 + 4tt .. +3] (w).
template <int NCOL>
__device__ __forceinline__ void prep_super_block(int sb, int m, int M, float4 v, float4 w,
                                                 int lane, uint2 *Bs, uint32_t *Bm, float *inv)
{
    const int cc = lane >> 3, tt = lane & 7;
    uint32_t mb = 0;
    mb = max(mb, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                     max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
    mb = max(mb, max(max(__float_as_uint(w.x) & 0x7fffffffu, __float_as_uint(w.y) & 0x7fffffffu),
                     max(__float_as_uint(w.z) & 0x7fffffffu, __float_as_uint(w.w) & 0x7fffffffu)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    // max|x| < 2^(eM+1): scaling by 2^(14-eM) keeps every term below 2^15.
    const int s = mb ? 14 - (int(mb >> 23) - 127) : 0;
    float xs[8] = {v.x, v.y, v.z, v.w, w.x, w.y, w.z, w.w};
    if (s >= -126 && s <= 127) {
        const float f = exp2i(s);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            xs[i] *= f;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            xs[i] = scale_pow2(xs[i], s);
    }
    __half hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        hi[i] = __float2half_rn(xs[i]);
        lo[i] = __float2half_rn(xs[i] - __half2float(hi[i]));
    }
    auto pack = [](__half a, __half b) {
        return uint32_t(__half_as_ushort(a)) | (uint32_t(__half_as_ushort(b)) << 16);
    };
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const size_t base = (size_t(sb) * 16 + 2 * tt + e) * NCOL;
        Bs[(base + 2 * m) * 4 + cc] = make_uint2(pack(hi[e], hi[e + 2]), pack(hi[4 + e], hi[6 + e]));
        Bs[(base + 2 * m + 1) * 4 + cc] =
            make_uint2(pack(lo[e], lo[e + 2]), pack(lo[4 + e], lo[6 + e]));
    }
    // Sub-block sums (sub-blocks 2cc and 2cc+1), fixed order over tt.
    float sl = (v.x + v.y) + (v.z + v.w);
    float sh = (w.x + w.y) + (w.z + w.w);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        sl += __shfl_xor_sync(0xffffffffu, sl, o);
        sh += __shfl_xor_sync(0xffffffffu, sh, o);
    }
    if (tt == 0) {
        // A sub-block sum of 32 terms below 2^15 stays below 2^20: a further
        // 2^-5 keeps it inside fp16 (undone exactly in the epilogue).
        const float a = scale_pow2(sl, s - 5), b = scale_pow2(sh, s - 5);
        const __half ah = __float2half_rn(a), bh = __float2half_rn(b);
        const __half al = __float2half_rn(a - __half2float(ah));
        const __half bl = __float2half_rn(b - __half2float(bh));
        Bm[(size_t(sb) * NCOL + 2 * m) * 4 + cc] = pack(ah, bh);
        Bm[(size_t(sb) * NCOL + 2 * m + 1) * 4 + cc] = pack(al, bl);
    }
    if (lane == 0)
        inv[sb * M + m] = scale_pow2(1.f, -s);
}

// One unit: a 16-row x 256-weight tile in shared memory (tp = the tile plus
// row g), this lane's chunk c, the B fragments of its super-block (bsb =
// Bs + ((sb*16)*NCOL + col)*4 + c), the min-MMA fragment bm and the inverse
// scale sc.  Adds this lane's two rows' contributions to tot0 / tot1.  Every
// load of the tile is consumed before returning.
template <int NCOL>
__device__ __forceinline__ void unit_dot(const uint8_t *tp, int c, uint32_t selA, uint32_t selB,
                                         bool hi4, const uint2 *bsb, uint32_t bm, float sc,
                                         float &tot0, float &tot1)
{
    const uint4 h0 = *reinterpret_cast<const uint4 *>(tp);
    const uint4 h1 = *reinterpret_cast<const uint4 *>(tp + 8 * 144);
    const uint4 qa0 = *reinterpret_cast<const uint4 *>(tp + 16 + 32 * c);
    const uint4 qa1 = *reinterpret_cast<const uint4 *>(tp + 32 + 32 * c);
    const uint4 qb0 = *reinterpret_cast<const uint4 *>(tp + 8 * 144 + 16 + 32 * c);
    const uint4 qb1 = *reinterpret_cast<const uint4 *>(tp + 8 * 144 + 32 + 32 * c);
    const RowScales r0 = row_scales(h0, selA, selB, hi4);
    const RowScales r1 = row_scales(h1, selA, selB, hi4);
    const uint32_t wa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
    const uint32_t wb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
    const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u, magic = 0x64006400u;
    float dq0[4], dq1[4];  // two independent accumulation chains (even / odd k-steps)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t xa = e ? (wa[t] >> 8) : wa[t];
            const uint32_t xb = e ? (wb[t] >> 8) : wb[t];
            const uint32_t a0 = hfma2(and_or(xa, mlo, magic), r0.SL, r0.CL);
            const uint32_t a1 = hfma2(and_or(xb, mlo, magic), r1.SL, r1.CL);
            const uint32_t a2 = hfma2(and_or(xa, mhi, magic), r0.SH, r0.CH);
            const uint32_t a3 = hfma2(and_or(xb, mhi, magic), r1.SH, r1.CH);
            const uint2 b = bsb[(2 * t + e) * NCOL * 4];
            float(&dq)[4] = e ? dq1 : dq0;
            if (t == 0)
                mma16816_zero(dq, a0, a1, a2, a3, b.x, b.y);
            else
                mma16816(dq, a0, a1, a2, a3, b.x, b.y);
        }
    }
    float dm[4];
    mma16816_zero(dm, r0.Am, r1.Am, 0u, 0u, bm, bm);
    tot0 = fmaf(fmaf(r0.d, (dq0[0] + dq1[0]) + (dq0[1] + dq1[1]),
                     -(r0.dmin * ((dm[0] + dm[1]) * 32.f))), sc, tot0);
    tot1 = fmaf(fmaf(r1.d, (dq0[2] + dq1[2]) + (dq0[3] + dq1[3]),
                     -(r1.dmin * ((dm[2] + dm[3]) * 32.f))), sc, tot1);
}

// ---------------------------------------------------------------------------
// One activation row: the nibbles enter the MMA as fp16 subnormals with no
// scale applied -- w & 0x000F000F is the half2 (q0, q1) * 2^-24 and
// w & 0x00F000F0 is (q0, q1) * 2^-20, both exact -- and each MMA gathers four
// sub-blocks, one per lane column c, so that the sub-block scales apply once
// per sub-block in fp32 instead of once per weight.
//
// MMA m = 2t + h of a unit (t = 0..7, h = 0 low / 1 high nibbles): lane c
// supplies word t of its chunk c, i.e. sub-block 2c+h, elements (4t, 4t+2)
// in k-slots (2c, 2c+1) and (4t+1, 4t+3) in k-slots (2c+8, 2c+9).  B column
// 2j holds the hi fp16 terms and column 2j+1 the lo terms of the activations
// of lane j's sub-block in lane j's k-slots, zeros elsewhere.  So lane c's
// accumulator columns (2c, 2c+1) are the hi and lo parts of the dot product
// of its rows with sub-block 2c+h; the 8 MMAs of each h accumulate a whole
// sub-block:
//   y_r += d * 2^-s * (sc_2c * 2^24 * D_lo[r] + sc_2c+1 * 2^20 * D_hi[r])
//          - dmin * (m_2c * X_2c + m_2c+1 * X_2c+1)
// with X_j the fp32 sum of sub-block j's activations and 2^s the exact
// power-of-two scale that puts the super-block's activations in fp16 range.
//
// B layout in shared memory: uint2 [super-block][m][c][part], part 0 = hi,
// 1 = lo; lane (g, c) with g >> 1 == c reads entry (c, g & 1), the other
// lanes a zero block laid out with the same stride.

struct SbScales {
    float sa, sb;    // sc_2c * 2^24, sc_2c+1 * 2^20
    float ma, mb;    // m_2c, m_2c+1
    float d, dmin;
};

__device__ __forceinline__ SbScales sb_scales(uint4 h, uint32_t selA, uint32_t selB, bool hi4)
{
    const uint32_t A = __byte_perm(h.y, h.z, selA);
    const uint32_t B = __byte_perm(h.w, h.w, selB);
    const uint32_t R = hi4 ? (((B & 0x00000F0Fu) | ((B >> 4) & 0x0F0F0000u)) |
                              ((A >> 2) & 0x30303030u))
                           : (A & 0x3F3F3F3Fu);  // bytes: sc_lo, sc_hi, m_lo, m_hi
    SbScales s;
    // (2^23 + v) * 2^k - 2^(23+k) = v * 2^k exactly.
    s.sa = fmaf(byte_magic(R, 0), 16777216.f, -140737488355328.f);  // 2^24, 2^47
    s.sb = fmaf(byte_magic(R, 1), 1048576.f, -8796093022208.f);     // 2^20, 2^43
    s.ma = byte_magic(R, 2) - 8388608.f;
    s.mb = byte_magic(R, 3) - 8388608.f;
    const float2 dd = half2_bits_to_float2(h.x);
    s.d = dd.x;
    s.dmin = dd.y;
    return s;
}

// Super-block sb of the activation row into the layout above.  Lane (cc, tt)
// = (lane >> 3, lane & 7) holds x[64cc + 4tt .. +3] (v, sub-block 2cc) and
// x[64cc + 32 + 4tt .. +3] (w, sub-block 2cc+1).  Bx: [NB][16][4][2] uint2,
// Xs: [NB][8] sub-block sums, inv: [NB] the inverse power-of-two scale.
__device__ __forceinline__ void prep_super_block_sb(int sb, float4 v, float4 w, int lane, uint2 *Bx,
                                                    float *Xs, float *inv)
{
    const int cc = lane >> 3, tt = lane & 7;
    uint32_t mb = 0;
    mb = max(mb, max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                     max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu)));
    mb = max(mb, max(max(__float_as_uint(w.x) & 0x7fffffffu, __float_as_uint(w.y) & 0x7fffffffu),
                     max(__float_as_uint(w.z) & 0x7fffffffu, __float_as_uint(w.w) & 0x7fffffffu)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    // max|x| < 2^(eM+1): scaling by 2^(14-eM) keeps every term below 2^15.
    const int s = mb ? 14 - (int(mb >> 23) - 127) : 0;
    float xs[8] = {v.x, v.y, v.z, v.w, w.x, w.y, w.z, w.w};
    if (s >= -126 && s <= 127) {
        const float f = exp2i(s);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            xs[i] *= f;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            xs[i] = scale_pow2(xs[i], s);
    }
    __half hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        hi[i] = __float2half_rn(xs[i]);
        lo[i] = __float2half_rn(xs[i] - __half2float(hi[i]));
    }
    auto pack = [](__half a, __half b) {
        return uint32_t(__half_as_ushort(a)) | (uint32_t(__half_as_ushort(b)) << 16);
    };
    // MMA 2tt + h takes elements (4tt, 4tt+2 | 4tt+1, 4tt+3) of sub-block 2cc+h.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int o = 4 * h;
        *reinterpret_cast<uint4 *>(Bx + ((size_t(sb) * 16 + 2 * tt + h) * 4 + cc) * 2) =
            make_uint4(pack(hi[o], hi[o + 2]), pack(hi[o + 1], hi[o + 3]), pack(lo[o], lo[o + 2]),
                       pack(lo[o + 1], lo[o + 3]));
    }
    // Sub-block sums (sub-blocks 2cc and 2cc+1), fixed order over tt.
    float sl = (v.x + v.y) + (v.z + v.w);
    float sh = (w.x + w.y) + (w.z + w.w);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        sl += __shfl_xor_sync(0xffffffffu, sl, o);
        sh += __shfl_xor_sync(0xffffffffu, sh, o);
    }
    if (tt == 0) {
        Xs[sb * 8 + 2 * cc] = sl;
        Xs[sb * 8 + 2 * cc + 1] = sh;
    }
    if (lane == 0)
        inv[sb] = scale_pow2(1.f, -s);
}

// One unit (16 rows x one super-block) for one activation row.  tp: the tile
// plus row g; bx: this lane's B entry of MMA 0 (consecutive MMAs 8 uint2
// apart); xab: (X_2c, X_2c+1); inv: 2^-s.  Adds the unit's share of rows g and
// g+8 over sub-blocks 2c and 2c+1 to tot0 / tot1 (the four lanes of a row
// pair are summed at the end of the row tile).
__device__ __forceinline__ void unit_dot_sb(const uint8_t *tp, int c, uint32_t selA, uint32_t selB,
                                            bool hi4, const uint2 *bx, float2 xab, float inv,
                                            float &tot0, float &tot1)
{
    const uint4 h0 = *reinterpret_cast<const uint4 *>(tp);
    const uint4 h1 = *reinterpret_cast<const uint4 *>(tp + 8 * 144);
    const uint4 qa0 = *reinterpret_cast<const uint4 *>(tp + 16 + 32 * c);
    const uint4 qa1 = *reinterpret_cast<const uint4 *>(tp + 32 + 32 * c);
    const uint4 qb0 = *reinterpret_cast<const uint4 *>(tp + 8 * 144 + 16 + 32 * c);
    const uint4 qb1 = *reinterpret_cast<const uint4 *>(tp + 8 * 144 + 32 + 32 * c);
    const uint32_t wa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
    const uint32_t wb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
    const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u;
    float dlo[4], dhi[4];  // sub-blocks 2c (low nibbles) and 2c+1 (high nibbles)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t xa = wa[t], xb = wb[t], ya = wa[t] >> 8, yb = wb[t] >> 8;
        const uint2 bl = bx[(2 * t) * 8], bh = bx[(2 * t + 1) * 8];
        if (t == 0) {
            mma16816_zero(dlo, xa & mlo, xb & mlo, ya & mlo, yb & mlo, bl.x, bl.y);
            mma16816_zero(dhi, xa & mhi, xb & mhi, ya & mhi, yb & mhi, bh.x, bh.y);
        } else {
            mma16816(dlo, xa & mlo, xb & mlo, ya & mlo, yb & mlo, bl.x, bl.y);
            mma16816(dhi, xa & mhi, xb & mhi, ya & mhi, yb & mhi, bh.x, bh.y);
        }
    }
    const SbScales r0 = sb_scales(h0, selA, selB, hi4);
    const SbScales r1 = sb_scales(h1, selA, selB, hi4);
    const float q0 = fmaf(r0.sa, dlo[0] + dlo[1], r0.sb * (dhi[0] + dhi[1]));
    const float q1 = fmaf(r1.sa, dlo[2] + dlo[3], r1.sb * (dhi[2] + dhi[3]));
    tot0 = fmaf(r0.d * inv, q0, fmaf(-r0.dmin, fmaf(r0.ma, xab.x, r0.mb * xab.y), tot0));
    tot1 = fmaf(r1.d * inv, q1, fmaf(-r1.dmin, fmaf(r1.ma, xab.x, r1.mb * xab.y), tot1));
}

// Lane-constant selectors of the (sc, m) bytes of chunk c (see the Q4_K
// packing): bytes (u0, u0+1) of sc12[0..3] and [4..7], and of sc12[8..11].
__device__ __forceinline__ void chunk_selectors(int c, uint32_t &selA, uint32_t &selB, bool &hi4)
{
    const uint32_t u0b = 2u * uint32_t(c & 1);
    selA = u0b * 0x1111u + 0x5410u;
    selB = u0b * 0x1111u + 0x1010u;
    hi4 = c >= 2;
}

// unit_dot for NT groups of four activation rows (B has NCOL = 8*NT columns):
// the A fragments of each k-step are built once and feed NT MMAs.  bsb =
// Bs + ((sb*16)*NCOL + g)*4 + c, bmp = Bm + (sb*NCOL + g)*4 + c, scp = inv +
// sb*4*NT + c (row 4*nt + c at scp[4*nt]).  tot0[nt] / tot1[nt] gain rows g
// and g+8 of activation row 4*nt + c.
template <int NT>
__device__ __forceinline__ void unit_dot_nt(const uint8_t *tp, int c, uint32_t selA, uint32_t selB,
                                            bool hi4, const uint2 *bsb, const uint32_t *bmp,
                                            const float *scp, float (&tot0)[NT], float (&tot1)[NT])
{
    constexpr int NCOL = 8 * NT;
    const uint4 h0 = *reinterpret_cast<const uint4 *>(tp);
    const uint4 h1 = *reinterpret_cast<const uint4 *>(tp + 8 * 144);
    const uint4 qa0 = *reinterpret_cast<const uint4 *>(tp + 16 + 32 * c);
    const uint4 qa1 = *reinterpret_cast<const uint4 *>(tp + 32 + 32 * c);
    const uint4 qb0 = *reinterpret_cast<const uint4 *>(tp + 8 * 144 + 16 + 32 * c);
    const uint4 qb1 = *reinterpret_cast<const uint4 *>(tp + 8 * 144 + 32 + 32 * c);
    const RowScales r0 = row_scales(h0, selA, selB, hi4);
    const RowScales r1 = row_scales(h1, selA, selB, hi4);
    const uint32_t wa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
    const uint32_t wb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
    const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u, magic = 0x64006400u;
    float dq[NT][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint32_t xa = e ? (wa[t] >> 8) : wa[t];
            const uint32_t xb = e ? (wb[t] >> 8) : wb[t];
            const uint32_t a0 = hfma2(and_or(xa, mlo, magic), r0.SL, r0.CL);
            const uint32_t a1 = hfma2(and_or(xb, mlo, magic), r1.SL, r1.CL);
            const uint32_t a2 = hfma2(and_or(xa, mhi, magic), r0.SH, r0.CH);
            const uint32_t a3 = hfma2(and_or(xb, mhi, magic), r1.SH, r1.CH);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint2 b = bsb[(2 * t + e) * NCOL * 4 + nt * 32];
                if (t == 0 && e == 0)
                    mma16816_zero(dq[nt], a0, a1, a2, a3, b.x, b.y);
                else
                    mma16816(dq[nt], a0, a1, a2, a3, b.x, b.y);
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint32_t bm = bmp[nt * 32];
        float dm[4];
        mma16816_zero(dm, r0.Am, r1.Am, 0u, 0u, bm, bm);
        const float sc = scp[4 * nt];
        tot0[nt] = fmaf(fmaf(r0.d, dq[nt][0] + dq[nt][1], -(r0.dmin * ((dm[0] + dm[1]) * 32.f))), sc,
                        tot0[nt]);
        tot1[nt] = fmaf(fmaf(r1.d, dq[nt][2] + dq[nt][3], -(r1.dmin * ((dm[2] + dm[3]) * 32.f))), sc,
                        tot1[nt]);
    }
}

} // namespace tc
} // namespace qmm
