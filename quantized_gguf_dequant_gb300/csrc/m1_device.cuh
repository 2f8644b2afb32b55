// m1_device.cuh -- device building blocks of the one-row Q4_K / Q5_K decode kernel
// (gemv_m1.cu): shared-memory and TMA helpers, the super-block header
// decode, the activation layout, and the arithmetic of one unit (16 rows x
// 256 weights) described at the top of gemv_m1.cu.
#pragma once

#include <cuda.h>

#include "qmm_device.cuh"
#include "tc_common.cuh"

namespace qmm {
namespace m1 {

using namespace tc;

constexpr int kMaxSlots = 16;  // ring slots at most

__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// One box of the 3-D column view (tmap.cu, make_q4k_column_map): rows
// [row, row+16) x super-blocks [sb, sb+WS) -> WS units of 16 x 144 bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int row, int sb,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(sb), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

// Shared-memory float load / store executed only where pred holds (the
// load gives 0 elsewhere).
__device__ __forceinline__ float lds_f32_if(uint32_t a, bool pred)
{
    float v = 0.f;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p ld.shared.f32 %0, [%1];\n\t}"
                 : "+f"(v)
                 : "r"(a), "r"(uint32_t(pred))
                 : "memory");
    return v;
}

__device__ __forceinline__ void sts_f32_if(uint32_t a, float v, bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.shared.f32 [%0], %1;\n\t}" ::"r"(a),
                 "f"(v), "r"(uint32_t(pred))
                 : "memory");
}

// Poll an mbarrier phase without spinning hard: between polls the thread
// sleeps, so a waiting producer leaves the issue slots to the consumers.
// Gives up (false) after `budget` cycles.
__device__ __forceinline__ bool mbar_wait_polled(uint64_t *bar, unsigned parity,
                                                 long long budget = kWaitBudgetCycles)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(128);
        if (mbar_try_wait(bar, parity))
            return true;
        if (clock64() - t0 > budget)
            return false;
    }
}

// Lane-constant part of the (sc, m) byte extraction for chunk c (see the
// Q4_K packing): sel picks bytes (u, u+1, 4+u, 5+u), u = 2*(c & 1).  For
// chunks 0 and 1 the fields are the low six bits of sc12[u..] and sc12[4+u..];
// for chunks 2 and 3 the low four bits come from sc12[8+u..] (low or high
// nibble) and the top two from bits 6-7 of sc12[u..] / sc12[4+u..].
struct ScaleSel {
    uint32_t sel, m1, m2, sh;
};

__device__ __forceinline__ ScaleSel scale_sel(int c)
{
    ScaleSel s;
    const uint32_t u = 2u * uint32_t(c & 1);
    s.sel = u * 0x1111u + 0x5410u;
    const bool hi = c >= 2;
    s.m1 = hi ? 0x0F0F0F0Fu : 0u;
    s.m2 = hi ? 0x30303030u : 0x3F3F3F3Fu;
    s.sh = hi ? 2u : 0u;
    return s;
}

// Bytes (sc_2c, sc_2c+1, m_2c, m_2c+1) of a row header.
__device__ __forceinline__ uint32_t scale_bytes(uint4 h, const ScaleSel &L)
{
    const uint32_t A = __byte_perm(h.y, h.z, L.sel);
    const uint32_t Q = __byte_perm(h.w, h.w >> 4, L.sel);
    return (Q & L.m1) | ((A >> L.sh) & L.m2);
}

// The contributions of rows g (header h0) and g+8 (h1) over this lane's two
// sub-blocks, in packed fp32: Dlo / Dhi hold (row g, row g+8) sums of the hi
// and lo MMA columns of sub-blocks 2c / 2c+1.
__device__ __forceinline__ float2 pair_total(uint4 h0, uint4 h1, const ScaleSel &L, float2 Dlo,
                                             float2 Dhi, float2 X0, float2 X1, float2 iv)
{
    const uint32_t R0 = scale_bytes(h0, L), R1 = scale_bytes(h1, L);
    // (2^23 + v) * 2^k - 2^(23+k) = v * 2^k exactly.
    const float2 sa = __ffma2_rn(make_float2(byte_magic(R0, 0), byte_magic(R1, 0)),
                                 make_float2(16777216.f, 16777216.f),
                                 make_float2(-140737488355328.f, -140737488355328.f));
    const float2 sb = __ffma2_rn(make_float2(byte_magic(R0, 1), byte_magic(R1, 1)),
                                 make_float2(1048576.f, 1048576.f),
                                 make_float2(-8796093022208.f, -8796093022208.f));
    const float2 ma = __fadd2_rn(make_float2(byte_magic(R0, 2), byte_magic(R1, 2)),
                                 make_float2(-8388608.f, -8388608.f));
    const float2 mb = __fadd2_rn(make_float2(byte_magic(R0, 3), byte_magic(R1, 3)),
                                 make_float2(-8388608.f, -8388608.f));
    const float2 d0 = half2_bits_to_float2(h0.x), d1 = half2_bits_to_float2(h1.x);
    const float2 q = __ffma2_rn(sa, Dlo, __fmul2_rn(sb, Dhi));
    const float2 mn = __ffma2_rn(ma, X0, __fmul2_rn(mb, X1));
    const float2 dd = __fmul2_rn(make_float2(d0.x, d1.x), iv);
    return __ffma2_rn(dd, q, __fmul2_rn(make_float2(-d0.y, -d1.y), mn));
}

// Activations of one super-block into its B entries bx[t][c][term] (uint4:
// the fragments of the low- and high-nibble MMAs of k-step t), its eight
// sub-block sums and 2^-s.  Lane (cc, tt) = (lane >> 3, lane & 7) holds
// x[64cc + 4tt .. +3] (v, sub-block 2cc) and x[64cc + 32 + 4tt .. +3] (w,
// sub-block 2cc+1).
// MODE 0: Q4_K / Q5_K (above).  MODE 1: Q6_K -- sums of the 16-weight
// groups instead (v's and w's halves).  MODE 2: IQ4_NL -- the k-slots of a
// lane column take adjacent weights ((v.x, v.y) in (2c, 2c+1), (v.z, v.w) in
// (2c+8, 2c+9); w likewise for the high-nibble MMA) and the sums are of the
// 32-weight blocks (v and w of lanes tt & ~3 .. tt | 3).  MODE 3: Q8_0 --
// MODE 2's adjacent k-slots with MODE 0's sums (v: block 2cc, w: 2cc+1).
template <int MODE = 0>
__device__ __forceinline__ void prep_sb(float4 v, float4 w, int lane, uint4 *bx, float *xsum,
                                        float *inv)
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
    if constexpr (MODE >= 2) {
        // k-step tt: elements (0, 1) in k-slots (2c, 2c+1), (2, 3) in (2c+8, 2c+9).
        bx[(tt * 4 + cc) * 2 + 0] = make_uint4(pack(hi[0], hi[1]), pack(hi[2], hi[3]),
                                               pack(hi[4], hi[5]), pack(hi[6], hi[7]));
        bx[(tt * 4 + cc) * 2 + 1] = make_uint4(pack(lo[0], lo[1]), pack(lo[2], lo[3]),
                                               pack(lo[4], lo[5]), pack(lo[6], lo[7]));
    } else {
        // k-step tt: elements (4tt, 4tt+2) in k-slots (2c, 2c+1), (4tt+1, 4tt+3) in (2c+8, 2c+9).
        bx[(tt * 4 + cc) * 2 + 0] = make_uint4(pack(hi[0], hi[2]), pack(hi[1], hi[3]),
                                               pack(hi[4], hi[6]), pack(hi[5], hi[7]));
        bx[(tt * 4 + cc) * 2 + 1] = make_uint4(pack(lo[0], lo[2]), pack(lo[1], lo[3]),
                                               pack(lo[4], lo[6]), pack(lo[5], lo[7]));
    }
    float sl = (v.x + v.y) + (v.z + v.w);
    float sh = (w.x + w.y) + (w.z + w.w);
    if constexpr (MODE == 2) {
        // Block sums (blocks 2cc and 2cc+1), fixed order.
        float sb = sl + sh;
#pragma unroll
        for (int o = 1; o < 4; o <<= 1)
            sb += __shfl_xor_sync(0xffffffffu, sb, o);
        if ((tt & 3) == 0)
            xsum[2 * cc + (tt >> 2)] = sb;
    } else if constexpr (MODE == 0 || MODE == 3) {
        // Sub-block sums (sub-blocks 2cc and 2cc+1), fixed order over tt.
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            sl += __shfl_xor_sync(0xffffffffu, sl, o);
            sh += __shfl_xor_sync(0xffffffffu, sh, o);
        }
        if (tt == 0) {
            xsum[2 * cc] = sl;
            xsum[2 * cc + 1] = sh;
        }
    } else {
        // Sums of the 16-weight groups (Q6_K's scale groups): lanes tt < 4
        // and tt >= 4 hold the two halves of v and of w; fixed order.
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            sl += __shfl_xor_sync(0xffffffffu, sl, o);
            sh += __shfl_xor_sync(0xffffffffu, sh, o);
        }
        if ((tt & 3) == 0) {
            const int g0 = 8 * (cc >> 1) + 2 * (cc & 1) + (tt >> 2);
            xsum[g0] = sl;
            xsum[g0 + 4] = sh;
        }
    }
    if (lane == 0)
        *inv = scale_pow2(1.f, -s);
}


// One unit for one lane: the unit's bytes for rows g (h0, qa0, qa1) and g+8
// (h1, qb0, qb1) of lane (g, c), the lane's B fragments of the super-block,
// its sub-block sums and inverse scale.  Returns the lane's share after the
// four lanes of the row pair are summed: lanes c = 0 / 1 hold rows g / g+8
// (the same fixed order for every unit).
__device__ __forceinline__ float unit_rows(uint4 h0, uint4 h1, uint4 qa0, uint4 qa1, uint4 qb0,
                                           uint4 qb1, const uint4 (&B)[8], const ScaleSel &L,
                                           int c, float2 X0, float2 X1, float2 iv)
{
    const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u;
    const uint32_t wa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
    const uint32_t wb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
    // four accumulation chains (k-steps even / odd) for the MMA latency
    float dlo[2][4], dhi[2][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t xa = wa[t], xb = wb[t], ya = wa[t] >> 8, yb = wb[t] >> 8;
        float(&l)[4] = dlo[t & 1];
        float(&h)[4] = dhi[t & 1];
        if (t < 2) {
            mma16816_zero(l, xa & mlo, xb & mlo, ya & mlo, yb & mlo, B[t].x, B[t].y);
            mma16816_zero(h, xa & mhi, xb & mhi, ya & mhi, yb & mhi, B[t].z, B[t].w);
        } else {
            mma16816(l, xa & mlo, xb & mlo, ya & mlo, yb & mlo, B[t].x, B[t].y);
            mma16816(h, xa & mhi, xb & mhi, ya & mhi, yb & mhi, B[t].z, B[t].w);
        }
    }
    const float2 lo = __fadd2_rn(__fadd2_rn(make_float2(dlo[0][0], dlo[0][2]), make_float2(dlo[0][1], dlo[0][3])),
                                 __fadd2_rn(make_float2(dlo[1][0], dlo[1][2]), make_float2(dlo[1][1], dlo[1][3])));
    const float2 hi = __fadd2_rn(__fadd2_rn(make_float2(dhi[0][0], dhi[0][2]), make_float2(dhi[0][1], dhi[0][3])),
                                 __fadd2_rn(make_float2(dhi[1][0], dhi[1][2]), make_float2(dhi[1][1], dhi[1][3])));
    const float2 tot = pair_total(h0, h1, L, lo, hi, X0, X1, iv);
    const bool odd = c & 1;
    float keep = odd ? tot.y : tot.x;
    keep += __shfl_xor_sync(0xffffffffu, odd ? tot.x : tot.y, 1);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    return keep;
}

// unit_rows for Q5_K: the same operands with each code's fifth bit (qh
// bytes l of the super-block's 32: bit 2c for the low nibble of chunk byte
// 32c + l, bit 2c+1 for the high one) put above its nibble -- bit 4 of the
// low-nibble half (value q * 2^-24, q < 32) and bit 8 of the high-nibble
// half (value 16 q * 2^-24): still exact fp16 subnormals.  ha / hb: the 32
// qh bytes of rows g and g+8.
__device__ __forceinline__ float unit_rows5(uint4 h0, uint4 h1, uint4 qa0, uint4 qa1, uint4 qb0,
                                            uint4 qb1, uint4 ha0, uint4 ha1, uint4 hb0, uint4 hb1,
                                            const uint4 (&B)[8], const ScaleSel &L, int c,
                                            float2 X0, float2 X1, float2 iv)
{
    const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u;
    const uint32_t blo = 0x00100010u, bhi = 0x01000100u;
    const uint32_t wa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
    const uint32_t wb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
    const uint32_t va[8] = {ha0.x, ha0.y, ha0.z, ha0.w, ha1.x, ha1.y, ha1.z, ha1.w};
    const uint32_t vb[8] = {hb0.x, hb0.y, hb0.z, hb0.w, hb1.x, hb1.y, hb1.z, hb1.w};
    const int sh = 2 * c;
    float dlo[4], dhi[4];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t xa = wa[t], xb = wb[t], ya = wa[t] >> 8, yb = wb[t] >> 8;
        const uint32_t pa = va[t] >> sh, pb = vb[t] >> sh, qa = pa >> 8, qb = pb >> 8;
        const uint32_t a0 = (xa & mlo) | ((pa << 4) & blo), a1 = (xb & mlo) | ((pb << 4) & blo);
        const uint32_t a2 = (ya & mlo) | ((qa << 4) & blo), a3 = (yb & mlo) | ((qb << 4) & blo);
        const uint32_t b0 = (xa & mhi) | ((pa << 7) & bhi), b1 = (xb & mhi) | ((pb << 7) & bhi);
        const uint32_t b2 = (ya & mhi) | ((qa << 7) & bhi), b3 = (yb & mhi) | ((qb << 7) & bhi);
        if (t == 0) {
            mma16816_zero(dlo, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816_zero(dhi, b0, b1, b2, b3, B[t].z, B[t].w);
        } else {
            mma16816(dlo, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816(dhi, b0, b1, b2, b3, B[t].z, B[t].w);
        }
    }
    const float2 tot = pair_total(h0, h1, L, __fadd2_rn(make_float2(dlo[0], dlo[2]),
                                                          make_float2(dlo[1], dlo[3])),
                                  __fadd2_rn(make_float2(dhi[0], dhi[2]), make_float2(dhi[1], dhi[3])),
                                  X0, X1, iv);
    const bool odd = c & 1;
    float keep = odd ? tot.y : tot.x;
    keep += __shfl_xor_sync(0xffffffffu, odd ? tot.x : tot.y, 1);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    return keep;
}

// ---------------------------------------------------------------- Q6_K
// A Q6_K super-block (210 bytes: 128 bytes of low nibbles, 64 of 2-bit high
// parts, 16 int8 scales, fp16 d) is read like Q4_K's: lane column c takes
// low-nibble byte chunk c (ql bytes 32c .. 32c+31), whose low nibbles are
// weights 128n + 32s + l and high nibbles weights 128n + 64 + 32s + l
// (n = c >> 1, s = c & 1, l < 32), and the high parts of those weights from
// qh bytes 32n + l (bits 2s..2s+1 for the low nibble, 2s+4..2s+5 for the
// high one).  The six-bit code q enters the MMA as an fp16 subnormal like a
// Q4_K nibble (q * 2^-24 from the low nibble, 16 q * 2^-24 from the high
// one), and the MMAs of k-steps 0-3 and 4-7 (l < 16, l >= 16) accumulate
// apart: each of the lane's four accumulators is one 16-weight scale group.
// Super-blocks sit 210 bytes apart, so a unit starts m = 0, 2, .., 14 bytes
// past a 16-byte boundary (the same m for every unit a warp reads): each
// 32-byte field comes in as three 16-byte loads from the boundary below and
// is realigned by W4 = m / 4 words and a two-byte permute when m % 4 = 2.

__device__ __forceinline__ uint32_t lds_u16(uint32_t a)
{
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// Words 0..7 of the 32 bytes starting W4 words (+2 bytes with sel 0x5432)
// after the 16-byte-aligned address ab.
template <int W4>
__device__ __forceinline__ void q6_field(uint32_t ab, unsigned sel, uint32_t (&out)[8])
{
    const uint4 u0 = lds128(ab), u1 = lds128(ab + 16), u2 = lds128(ab + 32);
    const uint32_t w[12] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w, u2.x, u2.y, u2.z, u2.w};
#pragma unroll
    for (int k = 0; k < 8; ++k)
        out[k] = __byte_perm(w[W4 + k], w[W4 + k + 1], sel);
}

// The lane's low-nibble chunk and high parts of the super-block at smem
// address a (a % 16 == m, W4 = m / 4).
template <int W4>
__device__ __forceinline__ void q6_fields(uint32_t a, int c, unsigned sel, uint32_t (&ql)[8],
                                          uint32_t (&qh)[8])
{
    const uint32_t ab = a & ~15u;
    q6_field<W4>(ab + 32 * c, sel, ql);
    q6_field<W4>(ab + 128 + 32 * (c >> 1), sel, qh);
}

__device__ __forceinline__ void q6_load(uint32_t a, int c, uint32_t (&ql)[8], uint32_t (&qh)[8])
{
    const unsigned sel = (a & 2u) ? 0x5432u : 0x3210u;
    switch ((a >> 2) & 3u) {
    case 0: q6_fields<0>(a, c, sel, ql, qh); break;
    case 1: q6_fields<1>(a, c, sel, ql, qh); break;
    case 2: q6_fields<2>(a, c, sel, ql, qh); break;
    default: q6_fields<3>(a, c, sel, ql, qh); break;
    }
}

// One Q6_K unit for one lane: rows g (qa, ha; scale bytes sa = (group
// 8n+2s, 8n+2s+1, 8n+4+2s, 8n+5+2s) as a word; d0) and g+8 (qb, hb, sb, d1);
// X: the four groups' activation sums (the same for both rows).
__device__ __forceinline__ float unit_rows6(const uint32_t (&qa)[8], const uint32_t (&ha)[8],
                                            const uint32_t (&qb)[8], const uint32_t (&hb)[8],
                                            uint32_t sa, uint32_t sb, uint32_t dd,
                                            const uint4 (&B)[8], int c, float4 X, float2 iv)
{
    const uint32_t mlo = 0x000F000Fu, mhi = 0x00F000F0u;
    const uint32_t blo = 0x00300030u, bhi = 0x03000300u;
    const int sh = 2 * (c & 1);
    float la[4], lb[4], ua[4], ub[4];  // low / high nibbles, groups l < 16 (a) and l >= 16 (b)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t xa = qa[t], xb = qb[t], ya = xa >> 8, yb = xb >> 8;
        const uint32_t pa = ha[t] >> sh, pb = hb[t] >> sh;  // bits 0-1: low nibble's high part
        const uint32_t ra = pa >> 4, rb = pb >> 4;          // bits 0-1: high nibble's
        const uint32_t a0 = (xa & mlo) | ((pa << 4) & blo), a1 = (xb & mlo) | ((pb << 4) & blo);
        const uint32_t a2 = (ya & mlo) | ((pa >> 4) & blo), a3 = (yb & mlo) | ((pb >> 4) & blo);
        const uint32_t b0 = (xa & mhi) | ((ra << 8) & bhi), b1 = (xb & mhi) | ((rb << 8) & bhi);
        const uint32_t b2 = (ya & mhi) | (ra & bhi), b3 = (yb & mhi) | (rb & bhi);
        float(&dl)[4] = t < 4 ? la : lb;
        float(&dh)[4] = t < 4 ? ua : ub;
        if ((t & 3) == 0) {
            mma16816_zero(dl, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816_zero(dh, b0, b1, b2, b3, B[t].z, B[t].w);
        } else {
            mma16816(dl, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816(dh, b0, b1, b2, b3, B[t].z, B[t].w);
        }
    }
    // (row g, row g+8) sums of the hi and lo columns of each group
    const float2 Dla = __fadd2_rn(make_float2(la[0], la[2]), make_float2(la[1], la[3]));
    const float2 Dlb = __fadd2_rn(make_float2(lb[0], lb[2]), make_float2(lb[1], lb[3]));
    const float2 Dua = __fadd2_rn(make_float2(ua[0], ua[2]), make_float2(ua[1], ua[3]));
    const float2 Dub = __fadd2_rn(make_float2(ub[0], ub[2]), make_float2(ub[1], ub[3]));
    // int8 scales -> floats: (2^23 + 128 + sc) - (2^23 + 128)
    const uint32_t qa8 = sa ^ 0x80808080u, qb8 = sb ^ 0x80808080u;
    const float2 off = make_float2(-8388736.f, -8388736.f);
    const float2 s0 = __fadd2_rn(make_float2(byte_magic(qa8, 0), byte_magic(qb8, 0)), off);
    const float2 s1 = __fadd2_rn(make_float2(byte_magic(qa8, 1), byte_magic(qb8, 1)), off);
    const float2 s2 = __fadd2_rn(make_float2(byte_magic(qa8, 2), byte_magic(qb8, 2)), off);
    const float2 s3 = __fadd2_rn(make_float2(byte_magic(qa8, 3), byte_magic(qb8, 3)), off);
    // sum (q - 32) x per group = D * 2^24 (low) or D * 2^20 (high), times
    // 2^-s for the activation scale, minus 32 X
    const float2 lo = __ffma2_rn(s0, Dla, __fmul2_rn(s1, Dlb));
    const float2 hi = __ffma2_rn(s2, Dua, __fmul2_rn(s3, Dub));
    const float2 q = __ffma2_rn(lo, make_float2(16777216.f, 16777216.f),
                                __fmul2_rn(hi, make_float2(1048576.f, 1048576.f)));
    const float2 mn = __ffma2_rn(s0, make_float2(X.x, X.x),
                                 __ffma2_rn(s1, make_float2(X.y, X.y),
                                            __ffma2_rn(s2, make_float2(X.z, X.z),
                                                       __fmul2_rn(s3, make_float2(X.w, X.w)))));
    const float2 d = half2_bits_to_float2(dd);  // (d of row g, d of row g+8)
    const float2 tot = __ffma2_rn(__fmul2_rn(d, iv), q,
                                  __fmul2_rn(make_float2(-32.f * d.x, -32.f * d.y), mn));
    const bool odd = c & 1;
    float keep = odd ? tot.y : tot.x;
    keep += __shfl_xor_sync(0xffffffffu, odd ? tot.x : tot.y, 1);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    return keep;
}

// ---------------------------------------------------------------- IQ4_NL
// Eight 18-byte blocks (fp16 d, 16 code bytes: byte j holds the codes of
// weights j (low nibble) and j+16 (high)) make a 144-byte unit like Q4_K's.
// Lane column c takes blocks 2c (k-steps 0-3) and 2c+1 (4-7); k-step t reads
// code bytes j..j+3 (j = 4(t & 3)) of its block.  Each code is looked up as
// u = book + 128 (1 .. 241, an exact fp16 subnormal u * 2^-24): the low 16
// bits of a code word hold four codes in nibble order (low j, high j, low
// j+1, high j+1) and serve as the byte-permute selector directly (bit 3
// cleared; a sign-replicating permute of the word and the word shifted by 4
// gives the 0xFF mask of the codes >= 8 that picks the second table half).
// Per block: sum book x = sum u x - 128 X.
struct Iq4Book {
    uint32_t t0, t1, t2, t3;  // u of codes 0-3, 4-7, 8-11, 12-15
};

__device__ __forceinline__ uint32_t prmt_m(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// u of the four codes in the low 16 bits of q (selector nibbles) -> bytes
// (u0, u1, u2, u3) in that order; m: the word's codes >= 8 mask source.
__device__ __forceinline__ uint32_t iq4_look(const Iq4Book &bk, uint32_t sel, uint32_t mask)
{
    const uint32_t lo = __byte_perm(bk.t0, bk.t1, sel), hi = __byte_perm(bk.t2, bk.t3, sel);
    return (lo & ~mask) | (hi & mask);
}

// One IQ4_NL unit for one lane: wa / wb the nine words at byte 36c of rows g
// and g+8 (block 2c: d in the low half of word 0, codes from byte 2; block
// 2c+1: d in the high half of word 4, codes in words 5-8); X: the sums of
// blocks 2c and 2c+1.
__device__ __forceinline__ float unit_rows_iq4(const uint32_t (&wa)[9], const uint32_t (&wb)[9],
                                               const Iq4Book &bk, const uint4 (&B)[8], int c,
                                               float2 X, float2 iv)
{
    float la[4], lb[4], ua[4], ub[4];  // low / high codes of block 2c (a) and 2c+1 (b)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t qa = t < 4 ? __byte_perm(wa[t], wa[t + 1], 0x5432u) : wa[t + 1];
        const uint32_t qb = t < 4 ? __byte_perm(wb[t], wb[t + 1], 0x5432u) : wb[t + 1];
        // codes of bytes j, j+1 (A) and j+2, j+3 (B) of rows g and g+8
        const uint32_t qa4 = qa << 4, qb4 = qb << 4;
        const uint32_t oa0 = iq4_look(bk, qa & 0x7777u, prmt_m(qa4, qa, 0xd9c8u));
        const uint32_t oa1 = iq4_look(bk, (qa >> 16) & 0x7777u, prmt_m(qa4, qa, 0xfbeau));
        const uint32_t ob0 = iq4_look(bk, qb & 0x7777u, prmt_m(qb4, qb, 0xd9c8u));
        const uint32_t ob1 = iq4_look(bk, (qb >> 16) & 0x7777u, prmt_m(qb4, qb, 0xfbeau));
        // (u_j, u_j+1) and (u_j+2, u_j+3): low codes; the high ones (j+16 ..)
        const uint32_t a0 = __byte_perm(oa0, 0u, 0x4240u), a1 = __byte_perm(ob0, 0u, 0x4240u);
        const uint32_t a2 = __byte_perm(oa1, 0u, 0x4240u), a3 = __byte_perm(ob1, 0u, 0x4240u);
        const uint32_t b0 = __byte_perm(oa0, 0u, 0x4341u), b1 = __byte_perm(ob0, 0u, 0x4341u);
        const uint32_t b2 = __byte_perm(oa1, 0u, 0x4341u), b3 = __byte_perm(ob1, 0u, 0x4341u);
        float(&dl)[4] = t < 4 ? la : lb;
        float(&dh)[4] = t < 4 ? ua : ub;
        if ((t & 3) == 0) {
            mma16816_zero(dl, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816_zero(dh, b0, b1, b2, b3, B[t].z, B[t].w);
        } else {
            mma16816(dl, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816(dh, b0, b1, b2, b3, B[t].z, B[t].w);
        }
    }
    // (row g, row g+8): sum u x of each block (hi + lo columns, both nibbles)
    const float2 Sa = __fadd2_rn(__fadd2_rn(make_float2(la[0], la[2]), make_float2(la[1], la[3])),
                                 __fadd2_rn(make_float2(ua[0], ua[2]), make_float2(ua[1], ua[3])));
    const float2 Sb = __fadd2_rn(__fadd2_rn(make_float2(lb[0], lb[2]), make_float2(lb[1], lb[3])),
                                 __fadd2_rn(make_float2(ub[0], ub[2]), make_float2(ub[1], ub[3])));
    const float2 da = half2_bits_to_float2(__byte_perm(wa[0], wb[0], 0x5410u));  // d of block 2c
    const float2 db = half2_bits_to_float2(__byte_perm(wa[4], wb[4], 0x7632u));  // d of block 2c+1
    const float2 k24 = make_float2(16777216.f, 16777216.f);
    const float2 ta = __ffma2_rn(__fmul2_rn(Sa, iv), k24, make_float2(-128.f * X.x, -128.f * X.x));
    const float2 tb = __ffma2_rn(__fmul2_rn(Sb, iv), k24, make_float2(-128.f * X.y, -128.f * X.y));
    const float2 tot = __ffma2_rn(da, ta, __fmul2_rn(db, tb));
    const bool odd = c & 1;
    float keep = odd ? tot.y : tot.x;
    keep += __shfl_xor_sync(0xffffffffu, odd ? tot.x : tot.y, 1);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    return keep;
}

// ---------------------------------------------------------------- Q8_0
// Eight 34-byte blocks (fp16 d, 32 int8 codes) make a 272-byte unit of 256
// weights.  Lane column c takes blocks 2c (the "low" MMA of each k-step) and
// 2c+1 (the "high" one); k-step t reads codes 4t .. 4t+3 of each.  A code
// enters as u = q + 128 (one XOR flips the sign bits), two codes per fp16
// pair (u * 2^-24, exact subnormals).  Per block: sum q x = sum u x - 128 X.

// One Q8_0 unit for one lane: wa / wb the seventeen words at byte 68c of
// rows g and g+8 (block 2c: d in the low half of word 0, codes from byte 2;
// block 2c+1: d in the high half of word 8, codes in words 9-16); X: the
// sums of blocks 2c and 2c+1.
__device__ __forceinline__ float unit_rows_q8(const uint32_t (&wa)[17], const uint32_t (&wb)[17],
                                              const uint4 (&B)[8], int c, float2 X, float2 iv)
{
    float da4[4], db4[4];  // blocks 2c and 2c+1
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t pa = __byte_perm(wa[t], wa[t + 1], 0x5432u) ^ 0x80808080u;  // block 2c
        const uint32_t pb = __byte_perm(wb[t], wb[t + 1], 0x5432u) ^ 0x80808080u;
        const uint32_t qa = wa[9 + t] ^ 0x80808080u;  // block 2c+1
        const uint32_t qb = wb[9 + t] ^ 0x80808080u;
        const uint32_t a0 = __byte_perm(pa, 0u, 0x4140u), a1 = __byte_perm(pb, 0u, 0x4140u);
        const uint32_t a2 = __byte_perm(pa, 0u, 0x4342u), a3 = __byte_perm(pb, 0u, 0x4342u);
        const uint32_t b0 = __byte_perm(qa, 0u, 0x4140u), b1 = __byte_perm(qb, 0u, 0x4140u);
        const uint32_t b2 = __byte_perm(qa, 0u, 0x4342u), b3 = __byte_perm(qb, 0u, 0x4342u);
        if (t == 0) {
            mma16816_zero(da4, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816_zero(db4, b0, b1, b2, b3, B[t].z, B[t].w);
        } else {
            mma16816(da4, a0, a1, a2, a3, B[t].x, B[t].y);
            mma16816(db4, b0, b1, b2, b3, B[t].z, B[t].w);
        }
    }
    // (row g, row g+8): sum u x of each block (hi + lo columns)
    const float2 Sa = __fadd2_rn(make_float2(da4[0], da4[2]), make_float2(da4[1], da4[3]));
    const float2 Sb = __fadd2_rn(make_float2(db4[0], db4[2]), make_float2(db4[1], db4[3]));
    const float2 da = half2_bits_to_float2(__byte_perm(wa[0], wb[0], 0x5410u));  // d of block 2c
    const float2 db = half2_bits_to_float2(__byte_perm(wa[8], wb[8], 0x7632u));  // d of block 2c+1
    const float2 k24 = make_float2(16777216.f, 16777216.f);
    const float2 ta = __ffma2_rn(__fmul2_rn(Sa, iv), k24, make_float2(-128.f * X.x, -128.f * X.x));
    const float2 tb = __ffma2_rn(__fmul2_rn(Sb, iv), k24, make_float2(-128.f * X.y, -128.f * X.y));
    const float2 tot = __ffma2_rn(da, ta, __fmul2_rn(db, tb));
    const bool odd = c & 1;
    float keep = odd ? tot.y : tot.x;
    keep += __shfl_xor_sync(0xffffffffu, odd ? tot.x : tot.y, 1);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    return keep;
}

} // namespace m1
} // namespace qmm
