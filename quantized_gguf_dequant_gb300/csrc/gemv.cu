// gemv.cu -- decode GEMV y = W x with the GGUF blocks decoded in registers
// (Q4_K and Q8_0), the weights streamed through shared memory by the TMA
// engine, a deterministic split-K, and programmatic dependent launch.
//
// The operation: "Building a Rust Inference Engine That Matches Llama.cpp",
// "Where the wins came from" -- quantized weights never become a
// full-precision buffer; the dequant math happens inline in the dot product.
//
// Work decomposition.  A CTA owns a contiguous range of rows (ranges are
// balanced to within one row) and one K-slice.  Its rows stream into a ring
// of shared-memory stages by bulk copies (completion counted on a "full"
// mbarrier).  Every warp consumes; warp 0 is also the producer and epilogue:
// once every warp has released a stage (its "empty" mbarrier) it adds the
// per-warp partial sums of the stage's rows in a fixed order, stores them and
// refills the slot -- there is no CTA-wide barrier in the loop.  Warps form
// row teams: thread c of a team owns the 64-weight chunk c of the K-slice for the
// whole kernel -- its 64 activations are loaded once, pre-scaled, and kept
// in registers -- and a team takes RPG rows of every stage.  The RPG partial
// sums of a thread meet the team's other lanes in a shuffle reduce-scatter.
// With split-K, K-slices write partial rows to the workspace and the last
// CTA of a row range (atomic ticket) adds them in slice order, so results
// are bitwise repeatable.
//
// Q4_K decode without integer-to-float conversions.  For a nibble q sitting
// at bit p (p <= 20) of a 32-bit word, masking the word leaves the bit
// pattern q * 2^p, and a bit pattern v < 2^24 read as a float is exactly
// v * 2^-149 (a subnormal, or the smallest normal binade, whose spacing is
// the same).  So float(word & (15 << p)) = q * 2^(p-149) exactly, with one
// LOP3.  Each activation is pre-scaled by 2^(149-p-E) for the bit position p
// of the nibble it meets (E chosen per chunk from its largest |x| so that
// nothing overflows), and one packed fp32 FMA (FFMA2, Blackwell) multiplies
// the low and the high nibble of a byte -- sub-blocks 2c and 2c+1 -- by their
// activations at once.  Per sub-block the sum S is then scaled back:
// contribution = d*sc*S*2^E - dmin*m*X, X the plain sum of the sub-block's
// activations.
#include <cstdio>
#include <cstdlib>

#include "formats.cuh"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kMaxConsumers = 256;  // consumer threads per CTA
constexpr int kStageBytesTarget = 36864;
constexpr int kCtasPerSm = 1;  // leaves room for the next kernel's CTA (PDL prefetch)
constexpr int kStages = 3;

struct __align__(16) U4 {
    uint32_t a, b, c, d;
};

__device__ __forceinline__ U4 lds128(const uint8_t *p)
{
    return *reinterpret_cast<const U4 *>(p);
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// Where a global row lives: matrix index and row within it.
__device__ __forceinline__ int matrix_of(const GemvArgs &a, int64_t row)
{
    int m = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroup - 1; ++i)
        if (i < a.nmat - 1 && row >= a.row_end[i])
            m = i + 1;
    return m;
}

__device__ __forceinline__ int64_t row_start(const GemvArgs &a, int m)
{
    return m == 0 ? 0 : a.row_end[m - 1];
}

__device__ __forceinline__ void load_chunk_x(const float *xp, float (&lo)[32], float (&hi)[32])
{
    const float4 *xv = reinterpret_cast<const float4 *>(xp);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 a = __ldg(xv + i);
        const float4 b = __ldg(xv + 8 + i);
        lo[4 * i + 0] = a.x; lo[4 * i + 1] = a.y; lo[4 * i + 2] = a.z; lo[4 * i + 3] = a.w;
        hi[4 * i + 0] = b.x; hi[4 * i + 1] = b.y; hi[4 * i + 2] = b.z; hi[4 * i + 3] = b.w;
    }
}

// ----------------------------------------------------------------- Q4_K
// Packed pairs of floats travel as 64-bit integers so that a pair is one
// register pair from the load to the packed FMA (no re-pairing moves).
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    return (uint64_t(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }

__device__ __forceinline__ uint64_t ffma2_u64(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Both nibbles of byte k of w in place, as the float pair
// (q_lo * 2^(8k-149), q_hi * 2^(8k+4-149)): one 64-bit AND of {w, w}.
template <int K>
__device__ __forceinline__ uint64_t nibble_pair(uint64_t ww)
{
    constexpr uint64_t mask = (uint64_t(0xF0u << (8 * K)) << 32) | uint64_t(0x0Fu << (8 * K));
    return ww & mask;
}

struct Q4State {
    uint64_t xp[32];  // (low-nibble, high-nibble) pre-scaled activations, l = 0..31
    float2 X;         // plain sums of the two sub-block halves
    float p1, p2;     // 2^E = p1 * p2
    uint32_t selA, selB;
    bool hi4;         // the chunk's sub-blocks are 4..7 (split 6-bit fields)
    int hdr_off, qs_off;
};

__device__ __forceinline__ void q4_prologue(Q4State &st, const float *x, int64_t gchunk,
                                            int local_chunk, bool idle)
{
    const int c4 = int(gchunk & 3);
    const float4 *xv = reinterpret_cast<const float4 *>(x + (gchunk >> 2) * 256 + c4 * 64);
    uint32_t mbits = 0;
    float sl = 0.f, sh = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 a = idle ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldg(xv + i);
        const float4 b = idle ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldg(xv + 8 + i);
        st.xp[4 * i + 0] = pack2(a.x, b.x);
        st.xp[4 * i + 1] = pack2(a.y, b.y);
        st.xp[4 * i + 2] = pack2(a.z, b.z);
        st.xp[4 * i + 3] = pack2(a.w, b.w);
    }
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        mbits = max(mbits, uint32_t(st.xp[l]) & 0x7fffffffu);
        mbits = max(mbits, uint32_t(st.xp[l] >> 32) & 0x7fffffffu);
        sl += lo_of(st.xp[l]);
        sh += hi_of(st.xp[l]);
    }
    // Largest |x| < 2^(eM+1).  E = eM + 23 keeps every pre-scaled activation
    // below 2^127 and puts the largest product near 2^-19.  The pre-scale of a
    // nibble at bit p is 2^(149-p-E) = 2^(126-p-eM).
    const int eM = int(mbits >> 23) - 127;
    const int E = eM + 23;
    const bool one_step = (eM >= -1) && (eM <= 212);
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        const int k = l & 3;
        const int p = (k < 3) ? 8 * k : 0;  // byte 3 is shifted down by 24 first
        const int s_lo = 126 - p - eM, s_hi = s_lo - 4;
        const float xl = lo_of(st.xp[l]), xh = hi_of(st.xp[l]);
        st.xp[l] = one_step ? pack2(xl * exp2i(s_lo), xh * exp2i(s_hi))
                            : pack2(scale_pow2(xl, s_lo), scale_pow2(xh, s_hi));
    }
    st.X = make_float2(sl, sh);
    const int E1 = E / 2;
    st.p1 = exp2i(E1);
    st.p2 = exp2i(E - E1);
    // Scale/min bytes of sub-blocks 2c4, 2c4+1 (see the Q4_K packing).
    const uint32_t u0 = 2u * uint32_t(c4 & 1);
    st.selA = u0 | ((u0 + 1) << 4) | ((4 + u0) << 8) | ((5 + u0) << 12);
    st.selB = u0 | ((u0 + 1) << 4) | (u0 << 8) | ((u0 + 1) << 12);
    st.hi4 = c4 >= 2;
    // Idle lanes (past the end of the K-slice) read the slice's first block,
    // whose finite values times their zero activations contribute exactly 0.
    st.hdr_off = idle ? 0 : (local_chunk >> 2) * 144;
    st.qs_off = idle ? 16 : st.hdr_off + 16 + 32 * c4;
}

// Partial dot product of one row's chunk (64 weights) with the chunk's
// activations, in natural units.
__device__ __forceinline__ float q4_row(const Q4State &st, const uint8_t *row)
{
    const U4 h = lds128(row + st.hdr_off);
    const U4 q0 = lds128(row + st.qs_off);
    const U4 q1 = lds128(row + st.qs_off + 16);
    const uint32_t qw[8] = {q0.a, q0.b, q0.c, q0.d, q1.a, q1.b, q1.c, q1.d};
    uint64_t acc0 = 0, acc1 = 0;  // (+0.0f, +0.0f)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint64_t ww = (uint64_t(qw[t]) << 32) | qw[t];
        const uint32_t w3 = qw[t] >> 24;
        const uint64_t ww3 = (uint64_t(w3) << 32) | w3;
        uint64_t &acc = (t & 1) ? acc1 : acc0;
        acc = ffma2_u64(nibble_pair<0>(ww), st.xp[4 * t + 0], acc);
        acc = ffma2_u64(nibble_pair<1>(ww), st.xp[4 * t + 1], acc);
        acc = ffma2_u64(nibble_pair<2>(ww), st.xp[4 * t + 2], acc);
        acc = ffma2_u64(nibble_pair<0>(ww3), st.xp[4 * t + 3], acc);
    }
    const float2 S = __fadd2_rn(make_float2(lo_of(acc0), hi_of(acc0)),
                                make_float2(lo_of(acc1), hi_of(acc1)));
    // (sc_lo, sc_hi, m_lo, m_hi) as bytes of R.
    const uint32_t A = __byte_perm(h.b, h.c, st.selA);
    const uint32_t B = __byte_perm(h.d, h.d, st.selB);
    const uint32_t R = st.hi4 ? (((B & 0x00000F0Fu) | ((B >> 4) & 0x0F0F0000u)) |
                                 ((A >> 2) & 0x30303030u))
                              : (A & 0x3F3F3F3Fu);
    const float2 magic = make_float2(-8388608.f, -8388608.f);
    const float2 sc = __fadd2_rn(make_float2(byte_magic(R, 0), byte_magic(R, 1)), magic);
    const float2 mm = __fadd2_rn(make_float2(byte_magic(R, 2), byte_magic(R, 3)), magic);
    const float2 us = __fmul2_rn(sc, S);
    const float2 vs = __fmul2_rn(mm, st.X);
    const float2 dd = half2_bits_to_float2(h.a);  // (d, dmin)
    const float t = (dd.x * (us.x + us.y)) * st.p1;
    return fmaf(t, st.p2, -(dd.y * (vs.x + vs.y)));
}

// ----------------------------------------------------------------- Q8_0
struct Q8State {
    float2 xp[32];  // (block A activation j, block B activation j)
    int off;        // byte offset of the chunk in a row
};

__device__ __forceinline__ void q8_prologue(Q8State &st, const float *x, int64_t gchunk,
                                            int local_chunk, bool idle)
{
    float a[32], b[32];
    if (idle) {
#pragma unroll
        for (int l = 0; l < 32; ++l)
            a[l] = b[l] = 0.f;
    } else {
        load_chunk_x(x + gchunk * 64, a, b);
    }
#pragma unroll
    for (int l = 0; l < 32; ++l)
        st.xp[l] = make_float2(a[l], b[l]);
    st.off = idle ? 0 : local_chunk * 68;
}

// Two Q8_0 blocks (68 bytes, 4-byte aligned): block A = bytes 0..33, block B
// = bytes 34..67.  int8 q -> float exactly: flip the sign bit (q + 128 as an
// unsigned byte), drop the byte into the mantissa of 2^23 and subtract
// 2^23 + 128.
__device__ __forceinline__ float q8_row(const Q8State &st, const uint8_t *row)
{
    const uint32_t *p = reinterpret_cast<const uint32_t *>(row + st.off);
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i)
        w[i] = p[i];
    const float2 d = half2_bits_to_float2(__byte_perm(w[0], w[8], 0x7610));
    const float2 off = make_float2(-8388736.f, -8388736.f);  // -(2^23 + 128)
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t qa = __funnelshift_r(w[k], w[k + 1], 16) ^ 0x80808080u;
        const uint32_t qb = w[9 + k] ^ 0x80808080u;
        float2 &acc = (k & 1) ? acc1 : acc0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 q = __fadd2_rn(make_float2(byte_magic(qa, i), byte_magic(qb, i)), off);
            acc = __ffma2_rn(q, st.xp[4 * k + i], acc);
        }
    }
    const float2 S = __fadd2_rn(acc0, acc1);
    return fmaf(d.x, S.x, d.y * S.y);
}

// ----------------------------------------------------------------- further formats
// Q5_K, Q6_K and IQ4_NL on the same staging and teams.  A thread's 64-weight
// chunk pairs weight l of its first half with weight l of its second half
// (xp[l] = (x_l, x_{32+l})), so that each packed FMA covers both.  Codes of
// up to 7 bits become the float 0.5 + b/256 with one byte permute (bytes
// [0, 0, b, 0x3f]); the group sums of x (prepared once) take the 0.5 back
// out, so no per-weight subtraction is needed.  IQ4_NL's signed book values
// go through 2^23 + 128 + v exactly.

__device__ __forceinline__ float half_plus(uint32_t v, int k)
{
    return __uint_as_float(__byte_perm(v, 0x3f000000u, 0x7054u | (unsigned(k) << 8)));
}

__device__ __forceinline__ uint32_t prmt_raw(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

struct FxState {
    float2 xp[32];  // (x_l, x_{32+l}) of the chunk
    float X[4];     // sums of x: Q5_K halves (X[0], X[1]); Q6_K the four groups of 16
    int off;        // byte offset of the chunk's unit (Q5_K, Q6_K) or blocks (IQ4_NL) in a row
    int c4;         // chunk within its super-block (K-quants)
};

template <int FMT>
__device__ __forceinline__ void fx_prologue(FxState &st, const float *x, int64_t gchunk,
                                            int local_chunk, bool idle)
{
    float a[32], b[32];
    if (idle) {
#pragma unroll
        for (int l = 0; l < 32; ++l)
            a[l] = b[l] = 0.f;
    } else {
        load_chunk_x(x + gchunk * 64, a, b);
    }
#pragma unroll
    for (int l = 0; l < 32; ++l)
        st.xp[l] = make_float2(a[l], b[l]);
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        s[0] += a[l];
        s[1] += a[16 + l];
        s[2] += b[l];
        s[3] += b[16 + l];
    }
    if (FMT == QMM_Q5_K) {
        st.X[0] = s[0] + s[1];
        st.X[1] = s[2] + s[3];
        st.X[2] = st.X[3] = 0.f;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st.X[i] = s[i];
    }
    st.c4 = int(gchunk & 3);
    if (FMT == QMM_Q5_K)
        st.off = idle ? 0 : (local_chunk >> 2) * 176;
    else if (FMT == QMM_Q6_K)
        st.off = idle ? 0 : (local_chunk >> 2) * 210;
    else
        st.off = idle ? 0 : local_chunk * 36;
}

// Q5_K: header, fifth bits and the chunk's nibbles, all 16-byte aligned.
__device__ __forceinline__ float q5_row(const FxState &st, const uint8_t *row)
{
    const uint8_t *u = row + st.off;
    const U4 h = lds128(u);
    const U4 h0 = lds128(u + 16), h1 = lds128(u + 32);
    const U4 q0 = lds128(u + 48 + 32 * st.c4), q1 = lds128(u + 64 + 32 * st.c4);
    const uint32_t qh[8] = {h0.a, h0.b, h0.c, h0.d, h1.a, h1.b, h1.c, h1.d};
    const uint32_t qs[8] = {q0.a, q0.b, q0.c, q0.d, q1.a, q1.b, q1.c, q1.d};
    const int j0 = 2 * st.c4;
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t hl = qh[t] >> j0;
        const uint32_t lo = (qs[t] & 0x0f0f0f0fu) | ((hl << 4) & 0x10101010u);
        const uint32_t hi = ((qs[t] >> 4) & 0x0f0f0f0fu) | ((hl << 3) & 0x10101010u);
        float2 &acc = (t & 1) ? acc1 : acc0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            acc = __ffma2_rn(make_float2(half_plus(lo, k), half_plus(hi, k)), st.xp[4 * t + k], acc);
    }
    const float2 S = __fadd2_rn(acc0, acc1);
    uint32_t sc0, m0, sc1, m1;
    {
        // the (sc, m) pairs of sub-blocks 2c4 and 2c4+1 (Q4_K packing)
        const int j1 = j0 + 1;
        auto sm = [&](int j, uint32_t &sc, uint32_t &m) {
            if (j < 4) {
                sc = (h.b >> (8 * j)) & 63u;
                m = (h.c >> (8 * j)) & 63u;
            } else {
                const int i = j - 4;
                const uint32_t bb = (h.d >> (8 * i)) & 0xffu;
                sc = (bb & 0x0fu) | (((h.b >> (8 * i + 6)) & 3u) << 4);
                m = (bb >> 4) | (((h.c >> (8 * i + 6)) & 3u) << 4);
            }
        };
        sm(j0, sc0, m0);
        sm(j1, sc1, m1);
    }
    const float2 dd = half2_bits_to_float2(h.a);  // (d, dmin)
    const float a0 = dd.x * float(sc0), a1 = dd.x * float(sc1);
    // a sum q x - b sum x, sum q x = 256 S - 128 X
    const float t = fmaf(256.f * a0, S.x, 256.f * a1 * S.y);
    const float c0 = fmaf(128.f, a0, dd.y * float(m0)), c1 = fmaf(128.f, a1, dd.y * float(m1));
    return t - fmaf(c0, st.X[0], c1 * st.X[1]);
}

// Q6_K: the unit is only 2-byte aligned; words are read from its start
// rounded down to 4 bytes and realigned with one byte permute each.
__device__ __forceinline__ float q6_row(const FxState &st, const uint8_t *row)
{
    const uintptr_t ua = reinterpret_cast<uintptr_t>(row + st.off);
    const uint32_t *wb = reinterpret_cast<const uint32_t *>(ua & ~uintptr_t(3));
    const unsigned sel = (ua & 2) ? 0x5432u : 0x3210u;
    auto U = [&](int k) { return __byte_perm(wb[k], wb[k + 1], sel); };
    const int n = st.c4 >> 1, odd = st.c4 & 1;
    const int t0 = 2 * odd;  // quarters t0 (weights 0..31) and t0 + 1 (32..63)
    float2 g01 = make_float2(0.f, 0.f), g23 = make_float2(0.f, 0.f);  // (group 0, 2), (1, 3)
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t qla = U(16 * n + m), qlb = U(16 * n + 8 + m), qh = U(32 + 8 * n + m);
        const uint32_t la = odd ? (qla >> 4) : qla, lb = odd ? (qlb >> 4) : qlb;
        const uint32_t qa = (la & 0x0f0f0f0fu) | (((qh >> (2 * t0)) & 0x03030303u) << 4);
        const uint32_t qb = (lb & 0x0f0f0f0fu) | (((qh >> (2 * t0 + 2)) & 0x03030303u) << 4);
        float2 &acc = (m < 4) ? g01 : g23;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            acc = __ffma2_rn(make_float2(half_plus(qa, k), half_plus(qb, k)), st.xp[4 * m + k], acc);
    }
    const uint32_t scw = U(48 + st.c4);  // the chunk's four int8 scales
    const uint32_t dw = (sel == 0x5432u) ? (wb[52] >> 16) : wb[52];
    const float d = __half2float(__ushort_as_half((unsigned short)(dw & 0xffffu)));
    // group g (16 weights): scale byte g; sum (q - 32) x = 256 S - 160 X
    const float s0 = d * float(int8_t(scw & 0xffu)), s1 = d * float(int8_t((scw >> 8) & 0xffu));
    const float s2 = d * float(int8_t((scw >> 16) & 0xffu)), s3 = d * float(int8_t(scw >> 24));
    float r = 256.f * (s0 * g01.x + s1 * g23.x + s2 * g01.y + s3 * g23.y);
    r -= 160.f * (s0 * st.X[0] + s1 * st.X[1] + s2 * st.X[2] + s3 * st.X[3]);
    return r;
}

// IQ4_NL: the chunk's two 18-byte blocks (4-byte aligned as a pair).
__device__ __forceinline__ float iq4_row(const FxState &st, const uint8_t *row)
{
    // the code book as int8 bytes: codes 0-7, 8-15
    constexpr uint32_t T0 = fmt::iq4nl_book_word(0), T1 = fmt::iq4nl_book_word(4),
                       T2 = fmt::iq4nl_book_word(8), T3 = fmt::iq4nl_book_word(12);
    const uint32_t *p = reinterpret_cast<const uint32_t *>(row + st.off);
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i)
        w[i] = p[i];
    const float2 d = half2_bits_to_float2(__byte_perm(w[0], w[4], 0x7610));  // (d_A, d_B)
    const float2 off = make_float2(-8388736.f, -8388736.f);                  // -(2^23 + 128)
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    // look four codes up: (book[c0], book[c1], book[c2], book[c3]) + 128 per byte
    auto look = [&](uint32_t codes) {  // codes: one 4-bit code per byte, in bits 0-3
        const uint32_t sel = codes & 0x0007u | (codes >> 4 & 0x0070u) | (codes >> 8 & 0x0700u) |
                             (codes >> 12 & 0x7000u);
        const uint32_t mask = prmt_raw(codes << 4, 0u, 0xba98u);  // 0xff where the code >= 8
        return ((__byte_perm(T0, T1, sel) & ~mask) | (__byte_perm(T2, T3, sel) & mask)) ^ 0x80808080u;
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ca = __byte_perm(w[i], w[i + 1], 0x5432u);  // block A code bytes 4i..4i+3
        const uint32_t cb = w[5 + i];                              // block B
        const uint32_t la = look(ca & 0x0f0f0f0fu), ha = look((ca >> 4) & 0x0f0f0f0fu);
        const uint32_t lb = look(cb & 0x0f0f0f0fu), hb = look((cb >> 4) & 0x0f0f0f0fu);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // weight 4i+k (low nibble) and 16+4i+k (high nibble) of each block
            const float2 vl = __fadd2_rn(make_float2(byte_magic(la, k), byte_magic(lb, k)), off);
            const float2 vh = __fadd2_rn(make_float2(byte_magic(ha, k), byte_magic(hb, k)), off);
            acc0 = __ffma2_rn(vl, st.xp[4 * i + k], acc0);
            acc1 = __ffma2_rn(vh, st.xp[16 + 4 * i + k], acc1);
        }
    }
    const float2 S = __fadd2_rn(acc0, acc1);
    return fmaf(d.x, S.x, d.y * S.y);
}

// ----------------------------------------------------------------- reduction
// Sum RPG values over groups of W lanes (W a power of two <= 32, RPG <= W)
// with a reduce-scatter: afterwards every lane holds the full sum of one of
// the RPG rows (its index is returned in j), and the lanes whose low
// log2(W/RPG) bits are zero are the designated writers.
template <int W, int RPG>
__device__ __forceinline__ float reduce_rows(const float (&v)[RPG], int lane, int &j)
{
    float cur[RPG];
#pragma unroll
    for (int k = 0; k < RPG; ++k)
        cur[k] = v[k];
    int idx = 0;
    int off = W / 2;
#pragma unroll
    for (int n = RPG; n > 1; n /= 2) {
        const int half = n / 2;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = upper ? cur[k] : cur[k + half];
            const float keep = upper ? cur[k + half] : cur[k];
            cur[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        if (upper)
            idx += half;
        off /= 2;
    }
#pragma unroll
    for (; off >= 1; off /= 2)
        cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], off);
    j = idx;
    return cur[0];
}

// ----------------------------------------------------------------- kernel
struct KParams {
    GemvArgs a;
    int kchunks, team, rg, stage_rows, stages, ksplit, row_slices;
    int64_t slice_bytes;
};

template <int FMT, int W, int RPG, int MINB>
__global__ void __launch_bounds__(kMaxConsumers, MINB) gemv_kernel(const __grid_constant__ KParams P)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const GemvArgs &a = P.a;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int NS = P.stages;
    const int SR = P.stage_rows;
    const int64_t SB = P.slice_bytes;
    const int rs = blockIdx.x / P.ksplit;  // row slice
    const int ks = blockIdx.x % P.ksplit;  // K-slice
    const int64_t base = a.N / P.row_slices, extra = a.N % P.row_slices;
    const int64_t r0 = rs * base + min64(rs, extra);
    const int64_t r1 = r0 + base + (rs < extra ? 1 : 0);
    const int nst = int((r1 - r0 + SR - 1) / SR);
    const int nwt = (P.team + 31) / 32;  // warps per team
    const int nwarps = int(blockDim.x) / 32;

    const size_t stage_bytes = size_t(SR) * size_t(SB);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(NS) * stage_bytes);
    uint64_t *empty = full + NS;
    float *red = reinterpret_cast<float *>(empty + NS);  // [NS][SR][nwt]

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], unsigned(nwarps));
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // Producer (lane 0 of warp 0): stage s goes to ring slot s % NS.
    const bool producer = tid < 32;
    uint64_t policy = 0;
    auto issue = [&](int s) {
        const int64_t ra = r0 + int64_t(s) * SR;
        const int64_t rb = min64(ra + SR, r1);
        uint8_t *dst = smem + size_t(s % NS) * stage_bytes;
        uint64_t *bar = &full[s % NS];
        mbar_arrive_expect_tx(bar, unsigned((rb - ra) * SB));
        if (P.ksplit == 1) {
            int64_t r = ra;
            while (r < rb) {
                const int m = matrix_of(a, r);
                const int64_t seg_end = min64(rb, a.row_end[m]);
                const uint8_t *src = a.w[m] + (r - row_start(a, m)) * a.row_bytes;
                bulk_g2s(dst + (r - ra) * SB, src, unsigned((seg_end - r) * a.row_bytes), bar,
                         policy);
                r = seg_end;
            }
        } else {
            for (int64_t r = ra; r < rb; ++r) {
                const int m = matrix_of(a, r);
                const uint8_t *src = a.w[m] + (r - row_start(a, m)) * a.row_bytes + int64_t(ks) * SB;
                bulk_g2s(dst + (r - ra) * SB, src, unsigned(SB), bar, policy);
            }
        }
    };
    // The weights are constant: the first stages are requested before waiting
    // for the previous kernel in the stream.
    int issued = min(NS, nst);
    if (tid == 0) {
        policy = policy_evict_first();
        for (int s = 0; s < issued; ++s)
            issue(s);
    }

    const int g = tid / P.team;  // row team
    const int c = tid % P.team;  // chunk lane within the team
    const bool idle = c >= P.kchunks;
    const int64_t gchunk = int64_t(ks) * P.kchunks + c;
    const int warp_in_team = c >> 5;
    const int rg = P.rg;

    pdl_wait();  // x, y and the workspace belong to the previous kernel until here
    Q4State s4;
    Q8State s8;
    FxState sx;
    if constexpr (FMT == QMM_Q4_K)
        q4_prologue(s4, a.x, gchunk, c, idle);
    else if constexpr (FMT == QMM_Q8_0)
        q8_prologue(s8, a.x, gchunk, c, idle);
    else
        fx_prologue<FMT>(sx, a.x, gchunk, c, idle);

    bool failed = false;
    for (int s = 0; s < nst; ++s) {
        const int b = s % NS;
        const unsigned parity = unsigned(s / NS) & 1u;
        if (!mbar_wait_bounded(&full[b], parity)) {
            failed = true;
            break;
        }
        const uint8_t *stage = smem + size_t(b) * stage_bytes;
        float part[RPG];
#pragma unroll
        for (int j = 0; j < RPG; ++j) {
            // Rows past the end of the range hold stale bytes; their sums are
            // computed and never stored.
            const uint8_t *row = stage + size_t(g + rg * j) * SB;
            if constexpr (FMT == QMM_Q4_K)
                part[j] = q4_row(s4, row);
            else if constexpr (FMT == QMM_Q8_0)
                part[j] = q8_row(s8, row);
            else if constexpr (FMT == QMM_Q5_K)
                part[j] = q5_row(sx, row);
            else if constexpr (FMT == QMM_Q6_K)
                part[j] = q6_row(sx, row);
            else
                part[j] = iq4_row(sx, row);
        }
        int j;
        const float v = reduce_rows<W, RPG>(part, lane, j);
        if ((lane & (W / RPG - 1)) == 0)
            red[(size_t(b) * SR + g + rg * j) * nwt + warp_in_team] = v;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[b]);
        if (producer) {
            // Epilogue of stage s once every warp has released it, then refill.
            if (!mbar_wait_bounded(&empty[b], parity)) {
                failed = true;
                break;
            }
            const int64_t ra = r0 + int64_t(s) * SR;
            const int nr = int(min64(SR, r1 - ra));
            const float *rd = red + size_t(b) * SR * nwt;
            for (int i = lane; i < nr; i += 32) {
                float acc = 0.f;
                for (int wv = 0; wv < nwt; ++wv)
                    acc += rd[i * nwt + wv];
                const int64_t row = ra + i;
                if (P.ksplit == 1) {
                    const int m = matrix_of(a, row);
                    a.y[m][row - row_start(a, m)] = acc;
                } else {
                    a.ws[int64_t(ks) * a.N + row] = acc;
                }
            }
            __syncwarp();
            if (issued < nst) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue(issued);
                }
                ++issued;
            }
        }
    }
    if (failed) {
        if (lane == 0)
            atomicOr(a.status, kStatusTimeoutBit);
        // Let the copies still in flight land before shared memory goes away.
        if (tid == 0)
            for (int s = 0; s < issued; ++s)
                mbar_wait_bounded(&full[s % NS], unsigned(s / NS) & 1u, 100000000ll);
        return;
    }
    if (producer && P.ksplit > 1) {
        __threadfence();
        __syncwarp();
        unsigned last = 0;
        if (lane == 0)
            last = atomicAdd(&a.tickets[rs], 1u) == unsigned(P.ksplit - 1);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            for (int64_t r = r0 + lane; r < r1; r += 32) {
                float acc = 0.f;
                for (int k = 0; k < P.ksplit; ++k)
                    acc += __ldcg(a.ws + int64_t(k) * a.N + r);
                const int m = matrix_of(a, r);
                a.y[m][r - row_start(a, m)] = acc;
            }
            if (lane == 0)
                a.tickets[rs] = 0u;
        }
    }
}

using KernelFn = void (*)(KParams);

template <int FMT, int W, int MINB>
KernelFn pick_rpg(int rpg)
{
    switch (rpg) {
    case 1: return gemv_kernel<FMT, W, 1, MINB>;
    case 2: return gemv_kernel<FMT, W, 2, MINB>;
    default: return gemv_kernel<FMT, W, 4, MINB>;
    }
}

template <int FMT, int MINB>
KernelFn pick_w(int w, int rpg)
{
    switch (w) {
    case 4: return pick_rpg<FMT, 4, MINB>(rpg);
    case 8: return pick_rpg<FMT, 8, MINB>(rpg);
    case 16: return pick_rpg<FMT, 16, MINB>(rpg);
    default: return pick_rpg<FMT, 32, MINB>(rpg);
    }
}

template <int FMT>
KernelFn pick(int w, int rpg, int minb)
{
    return minb >= 2 ? pick_w<FMT, 2>(w, rpg) : pick_w<FMT, 1>(w, rpg);
}

} // namespace

GemvPlan plan_gemv(int fmt, int64_t N, int64_t K, int sm_count, int force_ksplit)
{
    GemvPlan p;
    const int64_t chunks = K / 64;  // K % 256 == 0 for both formats here
    // A valid split cuts the row into equal slices of whole 256-weight blocks,
    // each at most kMaxConsumers chunks (one consumer thread per chunk).
    const int64_t nblocks = chunks / 4;
    auto valid = [&](int64_t ks) {
        return ks >= 1 && ks <= nblocks && nblocks % ks == 0 && chunks / ks <= kMaxConsumers;
    };
    int ksplit = int((chunks + kMaxConsumers - 1) / kMaxConsumers);
    while (!valid(ksplit))
        ++ksplit;
    // Tuning knobs (environment): CTAs per SM, stage size target in bytes,
    // ring depth.
    const char *e_cp = getenv("QMM_GEMV_CTAS_PER_SM");
    const char *e_sb = getenv("QMM_GEMV_STAGE_BYTES");
    const char *e_ns = getenv("QMM_GEMV_STAGES");
    const int ctas_per_sm = (e_cp && atoi(e_cp) > 0) ? atoi(e_cp) : kCtasPerSm;
    const int64_t target_ctas = int64_t(sm_count) * ctas_per_sm;
    while (force_ksplit <= 0 && N * ksplit < target_ctas && valid(int64_t(ksplit) * 2))
        ksplit *= 2;
    if (force_ksplit > 0 && valid(force_ksplit))
        ksplit = force_ksplit;
    p.ksplit = ksplit;
    p.kchunks = int(chunks / ksplit);
    int team = 4;
    if (p.kchunks <= 32) {
        while (team < p.kchunks)
            team *= 2;
    } else {
        team = (p.kchunks + 31) / 32 * 32;
    }
    p.rg = kMaxConsumers / team;
    if (p.rg < 1)
        p.rg = 1;
    p.threads = p.rg * team;
    // bytes of one row's K-slice: whole 256-weight groups of the format
    const int64_t group_bytes = fmt == QMM_Q4_K   ? 144
                                : fmt == QMM_Q5_K ? 176
                                : fmt == QMM_Q6_K ? 210
                                : fmt == QMM_IQ4_NL ? 144
                                                    : 272;
    p.slice_bytes = int64_t(p.kchunks / 4) * group_bytes;
    // Q8_0 rows are twice as long in bytes: a sweep of stage sizes and ring
    // depths on the Llama-3.1-8B Q8_0 step put two stages of four rows per
    // team (stage target >= 72 KB) first, 26 % ahead of the Q4_K setting.
    const int64_t stage_target = e_sb ? atoll(e_sb) : (fmt == QMM_Q8_0 ? 73728 : kStageBytesTarget);
    int rpg = int(stage_target / (int64_t(p.rg) * p.slice_bytes));
    const int wred = team < 32 ? team : 32;
    rpg = rpg >= 4 ? 4 : (rpg >= 2 ? 2 : 1);
    while (rpg > wred)
        rpg /= 2;
    p.rpg = rpg;
    p.stage_rows = p.rg * rpg;
    p.stages = e_ns ? atoi(e_ns) : (fmt == QMM_Q8_0 ? 2 : kStages);
    if (p.stages < 2)
        p.stages = 2;
    if (p.stages > 16)
        p.stages = 16;
    int64_t slices = target_ctas / ksplit;
    if (slices > N)
        slices = N;
    if (slices < 1)
        slices = 1;
    p.row_slices = int(slices);
    const int nwt = (team + 31) / 32;
    p.smem = size_t(p.stages) * size_t(p.stage_rows) * size_t(p.slice_bytes) +
             size_t(p.stages) * 16 + size_t(p.stages) * size_t(p.stage_rows) * nwt * 4;
    return p;
}

bool gemv_plan_takes(int fmt, const GemvPlan &p, int64_t row_bytes)
{
    if (fmt == QMM_Q4_K || fmt == QMM_Q8_0)
        return true;
    // The further formats: 32-lane teams only, and bulk copies need rows and
    // K-slices of whole 16-byte multiples (Q6_K: 2048 weights at a time).
    return p.threads / p.rg >= 32 && p.slice_bytes % 16 == 0 && row_bytes % 16 == 0;
}

size_t gemv_workspace_floats(const GemvPlan &p, int64_t N)
{
    return p.ksplit > 1 ? size_t(p.ksplit) * size_t(N) : 0;
}

cudaError_t launch_gemv(const GemvPlan &p, const GemvArgs &a, cudaStream_t s)
{
    KParams P;
    P.a = a;
    P.kchunks = p.kchunks;
    P.team = p.threads / p.rg;
    P.rg = p.rg;
    P.stage_rows = p.stage_rows;
    P.stages = p.stages;
    P.ksplit = p.ksplit;
    P.row_slices = p.row_slices;
    P.slice_bytes = p.slice_bytes;
    const int w = P.team < 32 ? P.team : 32;
    const char *e_lb = getenv("QMM_GEMV_MINB");
    const int minb = e_lb ? atoi(e_lb) : 1;
    KernelFn kern;
    switch (a.fmt) {
    case QMM_Q4_K: kern = pick<QMM_Q4_K>(w, p.rpg, minb); break;
    case QMM_Q8_0: kern = pick<QMM_Q8_0>(w, p.rpg, minb); break;
    case QMM_Q5_K: kern = pick_rpg<QMM_Q5_K, 32, 1>(p.rpg); break;
    case QMM_Q6_K: kern = pick_rpg<QMM_Q6_K, 32, 1>(p.rpg); break;
    default: kern = pick_rpg<QMM_IQ4_NL, 32, 1>(p.rpg); break;
    }
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), p.smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.row_slices * p.ksplit));
    cfg.blockDim = dim3(unsigned(p.threads));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, kern, P));
}

} // namespace qmm
