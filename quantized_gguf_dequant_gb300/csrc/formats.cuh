// formats.cuh -- the further GGUF block formats (Q5_K, Q6_K, IQ4_NL),
// decoded one 32-weight group at a time.  Each weight is the exact value of
// the format rounded once to fp32 (RN_fp32(w)), so the inspection path and
// the products see the same numbers.
//
// Layouts (GGUF block formats; little-endian):
//   Q5_K, 176 bytes / 256 weights: [fp16 d][fp16 dmin][12 bytes of 6-bit
//     scales and mins, the Q4_K packing][qh: 32 bytes of fifth bits]
//     [qs: 128 bytes of low nibbles, the Q4_K order].  Weight l (0..31) of
//     sub-block j: low four bits = nibble (j & 1) of qs[32*(j/2) + l], fifth
//     bit = bit j of qh[l].  w = d*sc_j*q - dmin*m_j: d*sc (17 bits) times q
//     (5 bits) and dmin*m (17 bits) are exact, fmaf rounds once.
//   Q6_K, 210 bytes / 256 weights: [ql: 128 bytes of low nibbles][qh: 64
//     bytes of 2-bit pairs][16 int8 scales][fp16 d].  Group j (weights
//     32j..32j+31): half n = j/4, quarter t = j%4; weight l has low bits =
//     nibble (t >= 2) of ql[64n + 32*(t & 1) + l], high bits = bits 2t, 2t+1
//     of qh[32n + l], scale = scales[2j + l/16]; w = d*scale*(q - 32).  d*scale
//     (19 bits) is exact, the product with q - 32 rounds once.
//   IQ4_NL, 18 bytes / 32 weights: [fp16 d][16 bytes]; weight l < 16 is the
//     low nibble of byte l, weight 16+l the high nibble; w = d*book[code],
//     exact (11 + 8 bits).
//   Q8_0, 34 bytes / 32 weights: [fp16 d][32 x int8]; w = d*q, exact.  Taken
//     here only for rows whose K is a multiple of 32 but not of 256 (the
//     other Q8_0 kernels take rows in whole 256-weight groups).
// Rows are whole blocks back to back; blocks are only 2-byte aligned (Q6_K,
// IQ4_NL, Q8_0), so the decoders read bytes.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "qmm.h"

namespace qmm {
namespace fmt {

constexpr int kQ80 = 8, kQ4K = 12, kQ5K = 13, kQ6K = 14, kIQ4NL = 20;

template <int F> struct Block;
template <> struct Block<kQ5K> { static constexpr int bytes = 176, weights = 256; };
template <> struct Block<kQ6K> { static constexpr int bytes = 210, weights = 256; };
template <> struct Block<kIQ4NL> { static constexpr int bytes = 18, weights = 32; };
template <> struct Block<kQ80> { static constexpr int bytes = 34, weights = 32; };

// The IQ4_NL code book: the value of each 4-bit code before the block scale
// (GGUF IQ4_NL format definition).
static __constant__ float kIq4nlBook[16] = {-127.f, -104.f, -83.f, -65.f, -49.f, -35.f,
                                            -22.f,  -10.f,  1.f,   13.f,  25.f,  38.f,
                                            53.f,   69.f,   89.f,  113.f};

// The same book as int8 bytes, four codes to a word (codes 0-3 in word 0,
// ...), for the kernels that look codes up with byte permutes.
constexpr int kIq4nlBookInt[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                   1,    13,   25,  38,  53,  69,  89,  113};
__host__ __device__ constexpr uint32_t iq4nl_book_word(int i)
{
    return uint32_t(kIq4nlBookInt[i] & 0xff) | (uint32_t(kIq4nlBookInt[i + 1] & 0xff) << 8) |
           (uint32_t(kIq4nlBookInt[i + 2] & 0xff) << 16) | (uint32_t(kIq4nlBookInt[i + 3] & 0xff) << 24);
}
static_assert(iq4nl_book_word(0) == 0xbfad9881u && iq4nl_book_word(12) == 0x71594535u,
              "IQ4_NL book packing");

__device__ __forceinline__ float half_bytes(const uint8_t *p)
{
    return __half2float(__ushort_as_half(uint16_t(p[0] | (p[1] << 8))));
}

// The 32 weights of group g (0 .. K/32 - 1) of a row, RN_fp32 of each.
template <int F>
__device__ __forceinline__ void decode_group(const uint8_t *row, int64_t g, float (&v)[32])
{
    if constexpr (F == kQ5K) {
        const uint8_t *blk = row + (g / 8) * 176;
        const int j = int(g % 8);
        const uint8_t *sc12 = blk + 4;
        int sc, m;
        if (j < 4) {
            sc = sc12[j] & 63;
            m = sc12[j + 4] & 63;
        } else {
            sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
            m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
        }
        const float a = half_bytes(blk) * float(sc);
        const float b = half_bytes(blk + 2) * float(m);
        const uint8_t *qh = blk + 16;
        const uint8_t *qs = blk + 48 + 32 * (j / 2);
        const int shift = (j & 1) ? 4 : 0;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const int q = ((qs[l] >> shift) & 15) | (((qh[l] >> j) & 1) << 4);
            v[l] = fmaf(a, float(q), -b);
        }
    } else if constexpr (F == kQ6K) {
        const uint8_t *blk = row + (g / 8) * 210;
        const int j = int(g % 8), n = j / 4, t = j % 4;
        const uint8_t *ql = blk + 64 * n + 32 * (t & 1);
        const uint8_t *qh = blk + 128 + 32 * n;
        const int lshift = t >= 2 ? 4 : 0;
        const float d = half_bytes(blk + 208);
        const float s0 = d * float(int8_t(blk[192 + 2 * j]));
        const float s1 = d * float(int8_t(blk[192 + 2 * j + 1]));
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const int q = ((ql[l] >> lshift) & 15) | (((qh[l] >> (2 * t)) & 3) << 4);
            v[l] = (l < 16 ? s0 : s1) * float(q - 32);
        }
    } else if constexpr (F == kQ80) {
        const uint8_t *blk = row + g * 34;
        const float d = half_bytes(blk);
#pragma unroll
        for (int l = 0; l < 32; ++l)
            v[l] = d * float(int8_t(blk[2 + l]));
    } else {
        const uint8_t *blk = row + g * 18;
        const float d = half_bytes(blk);
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            v[l] = d * kIq4nlBook[blk[2 + l] & 15];
            v[16 + l] = d * kIq4nlBook[blk[2 + l] >> 4];
        }
    }
}

} // namespace fmt
} // namespace qmm
