// formats_fast.cu -- decode GEMV (one activation row) for the further block
// formats Q5_K, Q6_K and IQ4_NL, at memory speed.
//
// The operation is the one of every path here ("Building a Rust Inference
// Engine That Matches Llama.cpp", "Where the wins came from": weights decoded
// inline in the dot product), for the formats "Frink Inference: the Rust
// alternative to llama.cpp" names ("Where Frink is already better than
// llama.cpp": the K-quants written byte-identically; "Where llama.cpp is
// still ahead": IQ4_NL).
//
// Layout of the work, as for the integer-dot kernel: a warp owns whole rows;
// each lane takes one 256-weight unit at a time (a Q5_K or Q6_K super-block,
// or eight IQ4_NL blocks), loads its bytes straight into registers and
// multiplies them with the activations, which the CTA keeps in shared
// memory.  Rows with 32 / 2^k units put several rows on one warp; longer
// rows have the lanes stride over the units.  Each row is reduced inside one
// warp by a fixed shuffle tree: results are bitwise repeatable.
//
// Per format:
//  Q5_K (176 bytes, 16-byte aligned): eleven 16-byte loads.  For four
//    weights of a sub-block, q = nibble | fifth bit << 4 is built for four
//    bytes at once; sum_l (a q_l - b) x_l = a * sum_l q_l x_l - b * sum_l x_l,
//    with a = d sc_j, b = dmin m_j exact in fp32 and the sub-block sums of x
//    prepared once per CTA.
//  Q6_K (210 bytes: only 2-byte aligned): 53 four-byte loads from the unit's
//    start rounded down to 4 bytes (no byte outside the unit is read), the
//    2-byte offset of odd units undone by one byte permute per word; per 16
//    weights the products (q - 32) x are summed and scaled by d * scale once.
//  IQ4_NL (eight 18-byte blocks = 144 bytes, 16-byte aligned): the 16-entry
//    code book is looked up four codes at a time with byte permutes over its
//    int8 values (codes 0-7 from the low half of the book, 8-15 from the high
//    half, chosen per byte by the code's top bit); per block the sum of
//    book[c] x is scaled by d.
// Integers become floats exactly through the 2^23 + b bit pattern.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "formats.cuh"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kWarpsF = 8;
constexpr int kUnitStride = 260;  // floats per 256-activation unit in shared memory

struct FmtParams {
    const uint8_t *w[kMaxGroup];
    float *y[kMaxGroup];
    int64_t row_end[kMaxGroup];
    int64_t N;          // rows of the whole group
    int64_t K;
    int NB;             // 256-weight units per row
    int64_t row_bytes;
    const float *x;     // M activation rows, ldx apart
    int64_t ldx;
    int M;              // activation rows of this pass (<= the kernel's MR)
    int64_t ldy;        // distance between a matrix's output rows
    int lshift;         // log2(lanes per row)
    int64_t n_groups;   // row groups (32 >> lshift rows each)
};

template <int F> struct Unit;
template <> struct Unit<fmt::kQ4K> { static constexpr int bytes = 144, words = 36; };
template <> struct Unit<fmt::kQ5K> { static constexpr int bytes = 176, words = 44; };
template <> struct Unit<fmt::kQ6K> { static constexpr int bytes = 210, words = 54; };
template <> struct Unit<fmt::kIQ4NL> { static constexpr int bytes = 144, words = 36; };

// Whether the next unit is loaded while the current one is used (two unit
// buffers in registers): Q6_K's 54-word unit stays single-buffered so that
// two CTAs fit an SM.
template <int F> constexpr bool kDoubleBuffer = F != fmt::kQ6K;

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The integer b (0..255) in byte k of v, as a float: the pattern 2^23 + b
// minus 2^23 (exact).  `bias` folds a constant offset into the subtraction.
__device__ __forceinline__ float byte_f(uint32_t v, int k, float bias)
{
    return __uint_as_float(__byte_perm(v, 0x4b000000u, 0x7540u | unsigned(k))) - bias;
}

// Load one unit's bytes as 32-bit words.  Q6_K: the 53 words from the unit's
// start rounded down to 4 bytes, and in word 53 the byte-permute selector
// that undoes the 2-byte offset of odd units (applied where the words are
// used).
template <int F>
__device__ __forceinline__ void load_unit(const uint8_t *a, uint32_t (&u)[Unit<F>::words])
{
    if constexpr (F == fmt::kQ6K) {
        const uint32_t *base = reinterpret_cast<const uint32_t *>(
            reinterpret_cast<uintptr_t>(a) & ~uintptr_t(3));
        const bool odd = (reinterpret_cast<uintptr_t>(a) & 3) != 0;
#pragma unroll
        for (int i = 0; i < 52; ++i)
            u[i] = __ldg(base + i);
        // the last word: bytes 206..209 of the unit (odd) or the two bytes
        // 208..209 (even), so nothing past the unit is read
        u[52] = odd ? __ldg(base + 52)
                    : uint32_t(__ldg(reinterpret_cast<const unsigned short *>(a + 208)));
        u[53] = odd ? 0x5432u : 0x3210u;
    } else {
#pragma unroll
        for (int i = 0; i < Unit<F>::words / 4; ++i) {
            const uint4 v = ldg_nc_v4(a + 16 * i);
            u[4 * i] = v.x;
            u[4 * i + 1] = v.y;
            u[4 * i + 2] = v.z;
            u[4 * i + 3] = v.w;
        }
    }
}

// prmt.b32 in its default mode, selector bit 3 included: a selector nibble
// 8 + i fills the output byte with the sign bit of source byte i (the
// __byte_perm intrinsic is specified on the low three bits only).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ float4 lds_f4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

__device__ __forceinline__ float half_lo(uint32_t w)
{
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}

// Byte k (0..127) of v as the float 0.5 + b/256: the pattern [0, 0, b, 0x3f]
// (exponent 2^-1, b in the top mantissa bits), one byte permute.  A sum of
// (0.5 + b/256) x over a group is 0.5 sum x + (1/256) sum b x; the group's
// sum of x is prepared once per CTA, so sum b x = 256 S - 128 sum x with no
// per-weight subtraction.  The offset costs about three bits of the fp32
// sum: far inside the 1e-4 bound for b up to 63.
__device__ __forceinline__ float half_plus(uint32_t v, int k)
{
    return __uint_as_float(__byte_perm(v, 0x3f000000u, 0x7054u | (unsigned(k) << 8)));
}

// s += (0.5 + b_k/256) * x_k for the four bytes of q and four activations.
__device__ __forceinline__ void fma4_half(uint32_t q, float4 xv, float2 &s)
{
    s = __ffma2_rn(make_float2(half_plus(q, 0), half_plus(q, 1)), make_float2(xv.x, xv.y), s);
    s = __ffma2_rn(make_float2(half_plus(q, 2), half_plus(q, 3)), make_float2(xv.z, xv.w), s);
}

// s += b_k * x_k for the four bytes of q (0..255, exact through 2^23 + b),
// four activations: every product exact, as the decode kernel's.
__device__ __forceinline__ void fma4_exact(uint32_t q, float4 xv, float2 &s)
{
    const float2 m = make_float2(-8388608.f, -8388608.f);
    const float2 a = __fadd2_rn(make_float2(byte_f(q, 0, 0.f), byte_f(q, 1, 0.f)), m);
    const float2 b = __fadd2_rn(make_float2(byte_f(q, 2, 0.f), byte_f(q, 3, 0.f)), m);
    s = __ffma2_rn(a, make_float2(xv.x, xv.y), s);
    s = __ffma2_rn(b, make_float2(xv.z, xv.w), s);
}

// acc[r] += sum_k w_k x_r,k over one unit, for MR activation rows; xs = the
// unit's 256 activations of row 0 in shared memory (row r at xs + r * xst),
// xsum = their group sums (Q5_K: 8 of 32, Q6_K: 16 of 16; row r at
// xsum + r * sst).  Every row's arithmetic is the same whatever MR is, so a
// row's result does not depend on how many rows share the pass.
template <int F, int MR>
__device__ __forceinline__ void unit_dot(const uint32_t (&u)[Unit<F>::words], const float *xs,
                                         int64_t xst, const float *xsum, int64_t sst,
                                         float (&acc)[MR])
{
    if constexpr (F == fmt::kQ5K || F == fmt::kQ4K) {
        // Q4_K is Q5_K without the fifth bits: its nibbles start at word 4
        constexpr int kQs = F == fmt::kQ5K ? 12 : 4;
        const float d = half_lo(u[0]), dmin = half_lo(u[0] >> 16);
        const uint32_t a = u[1], b = u[2], c = u[3];
        const uint32_t scA = a & 0x3f3f3f3fu, mA = b & 0x3f3f3f3fu;
        const uint32_t scB = (c & 0x0f0f0f0fu) | ((a >> 2) & 0x30303030u);
        const uint32_t mB = ((c >> 4) & 0x0f0f0f0fu) | ((b >> 2) & 0x30303030u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int sc = int(((j < 4 ? scA : scB) >> (8 * (j & 3))) & 0xffu);
            const int mn = int(((j < 4 ? mA : mB) >> (8 * (j & 3))) & 0xffu);
            float2 sv[MR];
#pragma unroll
            for (int r = 0; r < MR; ++r)
                sv[r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t qs = u[kQs + 8 * (j >> 1) + m];
                uint32_t q = (j & 1 ? qs >> 4 : qs) & 0x0f0f0f0fu;
                if constexpr (F == fmt::kQ5K)
                    q |= ((u[4 + m] >> j) & 0x01010101u) << 4;
#pragma unroll
                for (int r = 0; r < MR; ++r) {
                    if constexpr (F == fmt::kQ4K)
                        fma4_exact(q, lds_f4(xs + r * xst + 32 * j + 4 * m), sv[r]);
                    else
                        fma4_half(q, lds_f4(xs + r * xst + 32 * j + 4 * m), sv[r]);
                }
            }
            const float as = d * float(sc), bm = dmin * float(mn);
            if constexpr (F == fmt::kQ4K) {
                // a sum q x - b sum x, the products exact: a one-hot x gives
                // RN(a q - b), the exact weight rounded once
#pragma unroll
                for (int r = 0; r < MR; ++r) {
                    acc[r] = fmaf(as, sv[r].x + sv[r].y, acc[r]);
                    acc[r] = fmaf(-bm, xsum[r * sst + j], acc[r]);
                }
            } else {
                // a sum q x - b sum x with sum q x = 256 S - 128 sum x
                const float a256 = 256.f * as, c0 = -fmaf(128.f, as, bm);
#pragma unroll
                for (int r = 0; r < MR; ++r) {
                    acc[r] = fmaf(a256, sv[r].x + sv[r].y, acc[r]);
                    acc[r] = fmaf(c0, xsum[r * sst + j], acc[r]);
                }
            }
        }
    } else if constexpr (F == fmt::kQ6K) {
        const uint32_t sel = u[53];
        auto U = [&](int k) { return __byte_perm(u[k], u[k + 1], sel); };  // unit word k < 52
        const float d = half_lo(sel == 0x5432u ? (u[52] >> 16) : u[52]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // weights l = 16h .. 16h+15 of quarter t
                    float2 sv[MR];
#pragma unroll
                    for (int r = 0; r < MR; ++r)
                        sv[r] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const int m = 4 * h + mm;
                        const uint32_t ql = U(16 * n + 8 * (t & 1) + m), qh = U(32 + 8 * n + m);
                        const uint32_t q = ((t >= 2 ? ql >> 4 : ql) & 0x0f0f0f0fu) |
                                           (((qh >> (2 * t)) & 0x03030303u) << 4);
#pragma unroll
                        for (int r = 0; r < MR; ++r)
                            fma4_half(q, lds_f4(xs + r * xst + 128 * n + 32 * t + 4 * m), sv[r]);
                    }
                    const int si = 8 * n + 2 * t + h;  // scale index: weight / 16
                    const int sc = int(int8_t((U(48 + (si >> 2)) >> (8 * (si & 3))) & 0xffu));
                    // ds sum (q - 32) x = ds (256 S - 160 sum x)
                    const float ds = d * float(sc);
                    const float d256 = 256.f * ds, c0 = -160.f * ds;
#pragma unroll
                    for (int r = 0; r < MR; ++r) {
                        acc[r] = fmaf(d256, sv[r].x + sv[r].y, acc[r]);
                        acc[r] = fmaf(c0, xsum[r * sst + si], acc[r]);
                    }
                }
            }
        }
    } else {
        // the code book as int8 bytes: codes 0-7 in (T0, T1), 8-15 in (T2, T3)
        constexpr uint32_t T0 = fmt::iq4nl_book_word(0), T1 = fmt::iq4nl_book_word(4),
                           T2 = fmt::iq4nl_book_word(8), T3 = fmt::iq4nl_book_word(12);
        constexpr float kBias = 8388608.f + 128.f;  // 2^23 + 128: the int8 offset undone
        const float2 nb = make_float2(-kBias, -kBias);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int b0 = 18 * k;  // block byte offset within the unit
            const float d = (k & 1) ? half_lo(u[(b0 - 2) / 4] >> 16) : half_lo(u[b0 / 4]);
            float2 sv[MR];
#pragma unroll
            for (int r = 0; r < MR; ++r)
                sv[r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int o = b0 + 2 + 4 * p;  // byte offset of code bytes 4p..4p+3
                const uint32_t w = (o & 3) ? __byte_perm(u[o / 4], u[o / 4 + 1], 0x5432u) : u[o / 4];
                // codes in nibble order lo0 hi0 lo1 hi1 | lo2 hi2 lo3 hi3 =
                // weights 4p, 16+4p, 4p+1, 17+4p | 4p+2, 18+4p, 4p+3, 19+4p
                const uint32_t w4 = w << 4;
                const uint32_t sA = w & 0x7777u, sB = (w >> 16) & 0x7777u;
                const uint32_t mA = prmt(w4, w, 0xd9c8u), mB = prmt(w4, w, 0xfbeau);
                const uint32_t vA = (__byte_perm(T0, T1, sA) & ~mA) | (__byte_perm(T2, T3, sA) & mA);
                const uint32_t vB = (__byte_perm(T0, T1, sB) & ~mB) | (__byte_perm(T2, T3, sB) & mB);
                const uint32_t ua = vA ^ 0x80808080u, ub = vB ^ 0x80808080u;  // int8 + 128
                // low-nibble weights (4p .. 4p+3) and high-nibble ones (16+4p ..)
                const float2 l01 = __fadd2_rn(make_float2(byte_f(ua, 0, 0.f), byte_f(ua, 2, 0.f)), nb);
                const float2 l23 = __fadd2_rn(make_float2(byte_f(ub, 0, 0.f), byte_f(ub, 2, 0.f)), nb);
                const float2 h01 = __fadd2_rn(make_float2(byte_f(ua, 1, 0.f), byte_f(ua, 3, 0.f)), nb);
                const float2 h23 = __fadd2_rn(make_float2(byte_f(ub, 1, 0.f), byte_f(ub, 3, 0.f)), nb);
#pragma unroll
                for (int r = 0; r < MR; ++r) {
                    const float4 xl = lds_f4(xs + r * xst + 32 * k + 4 * p);
                    const float4 xh = lds_f4(xs + r * xst + 32 * k + 16 + 4 * p);
                    sv[r] = __ffma2_rn(l01, make_float2(xl.x, xl.y), sv[r]);
                    sv[r] = __ffma2_rn(l23, make_float2(xl.z, xl.w), sv[r]);
                    sv[r] = __ffma2_rn(h01, make_float2(xh.x, xh.y), sv[r]);
                    sv[r] = __ffma2_rn(h23, make_float2(xh.z, xh.w), sv[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < MR; ++r)
                acc[r] = fmaf(d, sv[r].x + sv[r].y, acc[r]);
        }
    }
}

template <int F, int MR>
__global__ void __launch_bounds__(32 * kWarpsF) gemv_fmt_fast_kernel(const __grid_constant__ FmtParams P)
{
    // [M][NB][kUnitStride] activations (each 256-weight unit's 256 values,
    // then 4 floats of padding so that lanes on neighbouring units read
    // different banks), then (Q5_K) [M][K/32] sums of 32
    extern __shared__ __align__(16) float sxf[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = 1 << P.lshift;
    const int sub = lane >> P.lshift, li = lane & (L - 1);
    const int64_t R = 32 >> P.lshift;
    const int64_t nw = int64_t(gridDim.x) * kWarpsF;
    const int spg = (P.NB + L - 1) / L;  // steps per row group: lane li takes unit li + L*step

    // The warp walks (row group, step) in order, loading the next position's
    // unit while it multiplies the current one (Q6_K: right after).  The
    // first unit is requested before the wait for the previous kernel.
    auto row_of = [&](int64_t g, int &mi, int64_t &lr) -> bool {
        const int64_t row = g * R + sub;
        if (row >= P.N)
            return false;
        mi = 0;
        while (row >= P.row_end[mi])
            ++mi;
        lr = row - (mi ? P.row_end[mi - 1] : 0);
        return true;
    };
    auto load = [&](int64_t g, int st, uint32_t (&u)[Unit<F>::words]) {
        int mi;
        int64_t lr;
        const int sb = li + L * st;
        if (g < P.n_groups && sb < P.NB && row_of(g, mi, lr))
            load_unit<F>(P.w[mi] + lr * P.row_bytes + int64_t(sb) * Unit<F>::bytes, u);
    };
    int64_t g = int64_t(blockIdx.x) * kWarpsF + warp;
    int st = 0;
    uint32_t ua[Unit<F>::words];
    load(g, st, ua);  // the weights do not depend on the previous kernel

    pdl_wait();  // x comes from the previous kernel
    pdl_launch_dependents();
    const int64_t xst = int64_t(P.NB) * kUnitStride;  // floats per activation row
    float *xsum = sxf + int64_t(MR) * xst;
    constexpr int G = F == fmt::kQ6K ? 16 : 32;  // group of the sums of x
    const int64_t ng = P.K / G;                   // groups per row
    // Stage the activations; the group sums come from neighbouring lanes'
    // float4 chunks (G / 4 lanes per group; K/4 is a multiple of 64, so
    // every warp runs the loop as a whole).
    const int64_t K4 = P.K / 4;
    for (int r = 0; r < P.M; ++r)
#pragma unroll 4
        for (int64_t i = threadIdx.x; i < K4; i += blockDim.x) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(P.x + r * P.ldx) + i);
            reinterpret_cast<float4 *>(sxf + r * xst + (i >> 6) * kUnitStride)[i & 63] = v;
            if constexpr (F != fmt::kIQ4NL) {
                float t = (v.x + v.y) + (v.z + v.w);
#pragma unroll
                for (int o = 1; o < G / 4; o <<= 1)
                    t += __shfl_xor_sync(0xffffffffu, t, o);
                if ((lane & (G / 4 - 1)) == 0)
                    xsum[r * ng + (4 * i) / G] = t;
            }
        }
    __syncthreads();

    float acc[MR];
#pragma unroll
    for (int r = 0; r < MR; ++r)
        acc[r] = 0.f;
    auto step = [&](uint32_t (&cur)[Unit<F>::words], uint32_t (&nxt)[Unit<F>::words]) {
        int64_t g2 = g;
        int st2 = st + 1;
        if (st2 == spg) {
            st2 = 0;
            g2 += nw;
        }
        if constexpr (kDoubleBuffer<F>)
            load(g2, st2, nxt);
        const int sb = li + L * st;
        int mi = 0;
        int64_t lr = 0;
        const bool have = row_of(g, mi, lr);
        if (have && sb < P.NB)
            unit_dot<F, MR>(cur, sxf + int64_t(sb) * kUnitStride, xst, xsum + (256 / G) * sb, ng,
                            acc);
        if (st == spg - 1) {
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                float a = acc[r];
                for (int o = L >> 1; o > 0; o >>= 1)
                    a += __shfl_xor_sync(0xffffffffu, a, o);
                if (li == 0 && have && r < P.M)
                    P.y[mi][r * P.ldy + lr] = a;
                acc[r] = 0.f;
            }
        }
        if constexpr (!kDoubleBuffer<F>)
            load(g2, st2, nxt);
        g = g2;
        st = st2;
    };
    if constexpr (kDoubleBuffer<F>) {
        uint32_t ub[Unit<F>::words];
        while (g < P.n_groups) {
            step(ua, ub);
            if (g >= P.n_groups)
                break;
            step(ub, ua);
        }
    } else {
        while (g < P.n_groups)
            step(ua, ua);  // the next unit is loaded after the current one is used
    }
}

template <int F, int MR>
cudaError_t launch_fast_t(const FmtParams &P, size_t smem, int sm_count, cudaStream_t s)
{
    const void *fn = reinterpret_cast<const void *>(gemv_fmt_fast_kernel<F, MR>);
    cudaError_t e = func_smem(fn, smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = func_occupancy(fn, 32 * kWarpsF, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    const int64_t want = (P.n_groups + kWarpsF - 1) / kWarpsF;
    const int64_t grid =
        std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sm_count) * std::max(per_sm, 1)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(32 * kWarpsF);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, gemv_fmt_fast_kernel<F, MR>, P));
}

template <int F>
cudaError_t launch_fast_f(const FmtParams &P, int MR, size_t smem, int sm_count, cudaStream_t s)
{
    if (MR == 4)
        return launch_fast_t<F, 4>(P, smem, sm_count, s);
    if (MR == 2)
        return launch_fast_t<F, 2>(P, smem, sm_count, s);
    return launch_fast_t<F, 1>(P, smem, sm_count, s);
}

} // namespace

size_t fmt_fast_smem(int fmt, int64_t K, int MR)
{
    const size_t sums = (fmt == fmt::kQ5K || fmt == fmt::kQ4K) ? size_t(K / 32)
                        : fmt == fmt::kQ6K                       ? size_t(K / 16)
                                                                 : 0;
    return size_t(MR) * (size_t(K / 256) * kUnitStride + sums) * 4;
}

int fmt_fast_rows(const Matrix &m, int M)
{
    if (!(m.fmt == fmt::kQ5K || m.fmt == fmt::kQ6K || m.fmt == fmt::kIQ4NL ||
          m.fmt == fmt::kQ4K) ||
        m.K % 256 != 0)
        return 0;
    const char *e = getenv("QMM_FMT_PATH");
    if (e && strcmp(e, "plain") == 0 && m.fmt != fmt::kQ4K)
        return 0;
    // rows per pass: 4, 2 or 1 -- the most that M has and shared memory holds
    for (int mr : {4, 2, 1})
        if ((mr <= M || mr == 1) && fmt_fast_smem(m.fmt, m.K, mr) <= size_t(227 * 1024))
            return mr;
    return 0;
}

cudaError_t launch_gemv_fmt_fast(const Matrix *const *ms, int n, const float *x, int64_t ldx,
                                 int M, float *const *ys, int64_t ldy, cudaStream_t s)
{
    const Matrix &m0 = *ms[0];
    const int MR = fmt_fast_rows(m0, M);
    if (MR == 0)
        return cudaErrorInvalidValue;
    FmtParams P;
    memset(&P, 0, sizeof(P));
    int64_t tot = 0;
    for (int i = 0; i < n; ++i) {
        P.w[i] = ms[i]->w;
        tot += ms[i]->N;
        P.row_end[i] = tot;
    }
    for (int i = n; i < kMaxGroup; ++i)
        P.row_end[i] = INT64_MAX;
    P.N = tot;
    P.K = m0.K;
    P.NB = int(m0.K / 256);
    P.row_bytes = m0.row_bytes;
    P.ldx = ldx;
    P.ldy = ldy;
    int lshift = 5;
    for (int l = 0; l <= 5; ++l)
        if ((1 << l) == P.NB)
            lshift = l;
    if (const char *e = getenv("QMM_FMT_LSHIFT"))  // tuning override: log2(lanes per row)
        lshift = std::min(5, std::max(0, atoi(e)));
    P.lshift = lshift;
    const int64_t R = 32 >> lshift;
    P.n_groups = (tot + R - 1) / R;
    const size_t smem = fmt_fast_smem(m0.fmt, m0.K, MR);
    // passes of MR rows (every row computed exactly as in a one-row pass)
    for (int r0 = 0; r0 < M; r0 += MR) {
        P.M = std::min(MR, M - r0);
        P.x = x + int64_t(r0) * ldx;
        for (int i = 0; i < n; ++i)
            P.y[i] = ys[i] + int64_t(r0) * ldy;
        cudaError_t e;
        switch (m0.fmt) {
        case fmt::kQ4K: e = launch_fast_f<fmt::kQ4K>(P, MR, smem, m0.sm_count, s); break;
        case fmt::kQ5K: e = launch_fast_f<fmt::kQ5K>(P, MR, smem, m0.sm_count, s); break;
        case fmt::kQ6K: e = launch_fast_f<fmt::kQ6K>(P, MR, smem, m0.sm_count, s); break;
        default: e = launch_fast_f<fmt::kIQ4NL>(P, MR, smem, m0.sm_count, s); break;
        }
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

} // namespace qmm
