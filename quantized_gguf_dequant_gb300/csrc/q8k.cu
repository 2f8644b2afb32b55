// q8k.cu -- the integer-dot variant: activations quantized to Q8_K, then a
// Q4_K GEMV whose inner products are integer dot products.
//
// "Frink Inference: the Rust alternative to llama.cpp", section "Where
// llama.cpp is still ahead": llama.cpp quantizes the activations to Q8_K
// before a K-quant dot product (Frink keeps them in f32, so the two engines'
// K-quant logits drift apart slightly).  This file is that path, as an
// opt-in next to the f32 one; the f32 path stays the default.
//
// Q8_K (GGUF): 256 activations per 292-byte block, [f32 d][256 x int8 q]
// [16 x int16 bsums], bsums[g] = q[16g] + ... + q[16g+15].  The block's max
// is the signed value of the first element of largest magnitude;
// iscale = -127 / max, q = min(127, round-half-even(iscale * x)),
// d = 1 / iscale, all in binary32 (zero block: d = 0, q = 0).
//
// Integer dot of one Q4_K super-block (d_w, dmin, eight 6-bit (sc_j, m_j),
// nibbles q_w) with one Q8_K block (d_x, q_x):
//   sum_k w_k * d_x q_x,k
//     = d_w d_x * sum_j sc_j * (sum_{k in j} q_w,k q_x,k)
//       - dmin d_x * sum_j m_j * (sum_{k in j} q_x,k)
// The inner sums are exact int32 (dp4a on four nibble bytes against four
// code bytes), the code sums come from bsums, and the two scale products are
// applied once per super-block in fp32.
//
// GEMV layout: one warp owns whole rows, so every output is reduced inside
// one warp in a fixed order (bitwise repeatable).  With 16 or fewer
// super-blocks per row that divide 32, the warp takes 32 / NB rows at once,
// one super-block per lane; otherwise its 32 lanes stride over the row's
// super-blocks.  A lane's super-block is 144 contiguous bytes, so a warp's
// nine 16-byte loads cover 32 neighbouring super-blocks (4.6 KB) and every
// byte fetched is used.  The Q8_K activations sit in shared memory, one
// 304-byte record per block: the 256 codes, the eight sub-block code sums
// (from bsums) and d.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kQ8kBlock = 292;   // bytes of one Q8_K block
constexpr int kRec = 304;        // shared-memory record per block (16-byte multiple)
constexpr int kWarps = 8;

// ------------------------------------------------------------------ quantize

// One warp per Q8_K block: lane l holds activations 4l..4l+3 and
// 128+4l..128+4l+3.
__global__ void __launch_bounds__(32 * kWarps) quantize_q8k_kernel(const float *__restrict__ x,
                                                                   int nb, uint8_t *out)
{
    pdl_wait();  // x may come from the previous kernel
    pdl_launch_dependents();
    const int b = int(blockIdx.x) * kWarps + int(threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= nb)
        return;
    const float *xb = x + int64_t(b) * 256;
    const float4 v0 = __ldg(reinterpret_cast<const float4 *>(xb) + lane);
    const float4 v1 = __ldg(reinterpret_cast<const float4 *>(xb + 128) + lane);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    // The first element of largest magnitude: within the lane in index
    // order, then across lanes (larger magnitude, or equal and earlier).
    float amax = 0.f, mx = 0.f;
    int mi = INT_MAX;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float ax = fabsf(v[k]);
        if (ax > amax) {
            amax = ax;
            mx = v[k];
            mi = (k < 4 ? 0 : 128) + 4 * lane + (k & 3);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oa = __shfl_xor_sync(0xffffffffu, amax, o);
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
        if (oa > amax || (oa == amax && oi < mi)) {
            amax = oa;
            mx = om;
            mi = oi;
        }
    }
    int q[8];
    float d = 0.f;
    if (amax == 0.f) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            q[k] = 0;
    } else {
        const float iscale = __fdiv_rn(-127.f, mx);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            q[k] = min(127, __float2int_rn(__fmul_rn(iscale, v[k])));
        d = __fdiv_rn(1.f, iscale);
    }
    uint8_t *ob = out + int64_t(b) * kQ8kBlock;
    const uint32_t w0 = (uint32_t(q[0]) & 0xffu) | ((uint32_t(q[1]) & 0xffu) << 8) |
                        ((uint32_t(q[2]) & 0xffu) << 16) | (uint32_t(q[3]) << 24);
    const uint32_t w1 = (uint32_t(q[4]) & 0xffu) | ((uint32_t(q[5]) & 0xffu) << 8) |
                        ((uint32_t(q[6]) & 0xffu) << 16) | (uint32_t(q[7]) << 24);
    reinterpret_cast<uint32_t *>(ob + 4)[lane] = w0;
    reinterpret_cast<uint32_t *>(ob + 4 + 128)[lane] = w1;
    if (lane == 0)
        *reinterpret_cast<float *>(ob) = d;
    // bsums: lanes 4g'..4g'+3 hold group g' (first half) and 8 + g' (second)
    int s0 = q[0] + q[1] + q[2] + q[3], s1 = q[4] + q[5] + q[6] + q[7];
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    if ((lane & 3) == 0) {
        int16_t *bs = reinterpret_cast<int16_t *>(ob + 260);
        bs[lane >> 2] = int16_t(s0);
        bs[8 + (lane >> 2)] = int16_t(s1);
    }
}

// ------------------------------------------------------------------ GEMV

struct Q8kParams {
    const uint8_t *w[kMaxGroup];
    float *y[kMaxGroup];
    int64_t row_end[kMaxGroup];  // cumulative row counts of the group
    int nmat;
    int64_t N;          // rows of the whole group
    int NB;             // super-blocks per row
    int64_t row_bytes;
    const uint8_t *xq;  // Q8_K blocks of the activations
    const float *x;     // or the f32 activations, quantized in the kernel
    int lshift;         // log2(lanes per row)
    int64_t n_groups;   // row groups (32 >> lshift rows each)
};

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ int byte_of(uint32_t v, int k) { return int((v >> (8 * k)) & 0xffu); }

// The integer dot of one Q4_K super-block (its nine 16-byte words) with one
// Q8_K record in shared memory, scaled: d_w d_x sumi - dmin d_x summ.
__device__ __forceinline__ float super_block_dot(const uint4 (&v)[9], const uint8_t *rec)
{
    const float2 dm = half2_bits_to_float2(v[0].x);  // (d, dmin)
    const uint32_t a = v[0].y, b = v[0].z, c = v[0].w;  // the twelve scale/min bytes
    // 6-bit (sc, m): j < 4 from the low six bits of bytes j and j+4; j >= 4
    // from the nibbles of byte j+4 and the top two bits of bytes j-4 and j
    const uint32_t scA = a & 0x3f3f3f3fu, mA = b & 0x3f3f3f3fu;
    const uint32_t scB = (c & 0x0f0f0f0fu) | ((a >> 2) & 0x30303030u);
    const uint32_t mB = ((c >> 4) & 0x0f0f0f0fu) | ((b >> 2) & 0x30303030u);
    const int *xs = reinterpret_cast<const int *>(rec + 256);  // code sums of the 8 sub-blocks
    int sumi = 0, summ = 0;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {  // 64 weights: sub-blocks 2ch (low nibbles), 2ch+1 (high)
        const uint4 q0 = v[1 + 2 * ch], q1 = v[2 + 2 * ch];
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint4 xl0 = lds128(rec + 64 * ch), xl1 = lds128(rec + 64 * ch + 16);
        const uint4 xh0 = lds128(rec + 64 * ch + 32), xh1 = lds128(rec + 64 * ch + 48);
        const uint32_t xl[8] = {xl0.x, xl0.y, xl0.z, xl0.w, xl1.x, xl1.y, xl1.z, xl1.w};
        const uint32_t xh[8] = {xh0.x, xh0.y, xh0.z, xh0.w, xh1.x, xh1.y, xh1.z, xh1.w};
        int dlo = 0, dhi = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            dlo = __dp4a(int(qw[m] & 0x0f0f0f0fu), int(xl[m]), dlo);
            dhi = __dp4a(int((qw[m] >> 4) & 0x0f0f0f0fu), int(xh[m]), dhi);
        }
        const int j0 = 2 * ch, j1 = 2 * ch + 1;
        const int sc0 = j0 < 4 ? byte_of(scA, j0) : byte_of(scB, j0 - 4);
        const int sc1 = j1 < 4 ? byte_of(scA, j1) : byte_of(scB, j1 - 4);
        const int m0 = j0 < 4 ? byte_of(mA, j0) : byte_of(mB, j0 - 4);
        const int m1 = j1 < 4 ? byte_of(mA, j1) : byte_of(mB, j1 - 4);
        sumi += sc0 * dlo + sc1 * dhi;
        summ += m0 * xs[j0] + m1 * xs[j1];
    }
    const float dx = *reinterpret_cast<const float *>(rec + 288);
    return (dm.x * dx) * float(sumi) - (dm.y * dx) * float(summ);
}

// Q8_K quantization of activation block b (256 values at xb) by one warp:
// the record's codes, sub-block code sums and d, exactly as
// quantize_q8k_kernel writes the block (the same steps and rounding).
__device__ __forceinline__ void quantize_record(const float *xb, int lane, uint8_t *rec)
{
    const float4 v0 = __ldg(reinterpret_cast<const float4 *>(xb) + lane);
    const float4 v1 = __ldg(reinterpret_cast<const float4 *>(xb + 128) + lane);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float amax = 0.f, mx = 0.f;
    int mi = INT_MAX;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float ax = fabsf(v[k]);
        if (ax > amax) {
            amax = ax;
            mx = v[k];
            mi = (k < 4 ? 0 : 128) + 4 * lane + (k & 3);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oa = __shfl_xor_sync(0xffffffffu, amax, o);
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
        if (oa > amax || (oa == amax && oi < mi)) {
            amax = oa;
            mx = om;
            mi = oi;
        }
    }
    int q[8];
    float d = 0.f;
    if (amax == 0.f) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            q[k] = 0;
    } else {
        const float iscale = __fdiv_rn(-127.f, mx);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            q[k] = min(127, __float2int_rn(__fmul_rn(iscale, v[k])));
        d = __fdiv_rn(1.f, iscale);
    }
    reinterpret_cast<uint32_t *>(rec)[lane] =
        (uint32_t(q[0]) & 0xffu) | ((uint32_t(q[1]) & 0xffu) << 8) |
        ((uint32_t(q[2]) & 0xffu) << 16) | (uint32_t(q[3]) << 24);
    reinterpret_cast<uint32_t *>(rec + 128)[lane] =
        (uint32_t(q[4]) & 0xffu) | ((uint32_t(q[5]) & 0xffu) << 8) |
        ((uint32_t(q[6]) & 0xffu) << 16) | (uint32_t(q[7]) << 24);
    // sub-block j (32 codes): lanes 8j'..8j'+7 of the first (j = j') or
    // second (j = 4 + j') half
    int s0 = q[0] + q[1] + q[2] + q[3], s1 = q[4] + q[5] + q[6] + q[7];
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    if ((lane & 7) == 0) {
        reinterpret_cast<int *>(rec + 256)[lane >> 3] = s0;
        reinterpret_cast<int *>(rec + 256)[4 + (lane >> 3)] = s1;
    }
    if (lane == 0)
        *reinterpret_cast<float *>(rec + 288) = d;
}

template <bool FROMX>
__global__ void __launch_bounds__(32 * kWarps) gemv_q8k_kernel(const __grid_constant__ Q8kParams P)
{
    extern __shared__ __align__(16) uint8_t sx[];
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = 1 << P.lshift;              // lanes per row
    const int sub = lane >> P.lshift, li = lane & (L - 1);
    const int64_t R = 32 >> P.lshift;         // rows per group
    const int64_t nw = int64_t(gridDim.x) * kWarps;
    const int spg = (P.NB + L - 1) / L;       // steps per group: lane li takes super-block li + L*step

    // The warp walks (group, step) in order; the weights of the next
    // position are loaded while the current one is computed.  The first
    // loads go out before the wait for the previous kernel: the weights do
    // not depend on it, the activations do.
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
    auto load = [&](int64_t g, int st, uint4 (&v)[9]) {
        int mi;
        int64_t lr;
        const int sb = li + L * st;
        if (g < P.n_groups && sb < P.NB && row_of(g, mi, lr)) {
            const uint4 *src =
                reinterpret_cast<const uint4 *>(P.w[mi] + lr * P.row_bytes + int64_t(sb) * 144);
#pragma unroll
            for (int i = 0; i < 9; ++i)
                v[i] = ldg_stream(src + i);
        }
    };

    int64_t g = int64_t(blockIdx.x) * kWarps + warp;
    int st = 0;
    uint4 va[9], vb[9];
    load(g, st, va);

    pdl_wait();  // the activations come from the previous kernel
    if constexpr (FROMX) {
        // Quantize the activations here, one Q8_K block per warp in turn.
        for (int b = warp; b < P.NB; b += kWarps)
            quantize_record(P.x + int64_t(b) * 256, lane, sx + b * kRec);
    } else {
    // Stage the activations: codes (4-byte words), sub-block code sums, d.
    for (int i = threadIdx.x; i < P.NB * 64; i += blockDim.x) {
        const int b = i >> 6, j = i & 63;
        reinterpret_cast<uint32_t *>(sx + b * kRec)[j] =
            __ldg(reinterpret_cast<const uint32_t *>(P.xq + int64_t(b) * kQ8kBlock + 4) + j);
    }
    for (int i = threadIdx.x; i < P.NB * 8; i += blockDim.x) {
        const int b = i >> 3, j = i & 7;
        const int16_t *bs = reinterpret_cast<const int16_t *>(P.xq + int64_t(b) * kQ8kBlock + 260);
        reinterpret_cast<int *>(sx + b * kRec + 256)[j] = int(bs[2 * j]) + int(bs[2 * j + 1]);
    }
    for (int b = threadIdx.x; b < P.NB; b += blockDim.x)
        *reinterpret_cast<float *>(sx + b * kRec + 288) =
            __ldg(reinterpret_cast<const float *>(P.xq + int64_t(b) * kQ8kBlock));
    }
    __syncthreads();

    float acc = 0.f;
    // One position: prefetch the next into `nxt`, add the current (`cur`),
    // and at a group's last step reduce the row and store it.
    auto step = [&](uint4 (&cur)[9], uint4 (&nxt)[9]) {
        int64_t g2 = g;
        int st2 = st + 1;
        if (st2 == spg) {
            st2 = 0;
            g2 += nw;
        }
        load(g2, st2, nxt);
        const int sb = li + L * st;
        int mi = 0;
        int64_t lr = 0;
        const bool have = row_of(g, mi, lr);
        if (have && sb < P.NB)
            acc += super_block_dot(cur, sx + sb * kRec);
        if (st == spg - 1) {
            for (int o = L >> 1; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (li == 0 && have)
                P.y[mi][lr] = acc;
            acc = 0.f;
        }
        g = g2;
        st = st2;
    };
    while (g < P.n_groups) {
        step(va, vb);
        if (g >= P.n_groups)
            break;
        step(vb, va);
    }
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return counted(cudaLaunchKernelEx(&cfg, k, args...));
}

} // namespace

size_t q8k_smem(int64_t K) { return size_t(K / 256) * kRec; }

cudaError_t launch_quantize_q8k(const float *x, int64_t K, uint8_t *out, cudaStream_t s)
{
    const int nb = int(K / 256);
    return launch_pdl(quantize_q8k_kernel, dim3(unsigned((nb + kWarps - 1) / kWarps)),
                      dim3(32 * kWarps), 0, s, x, nb, out);
}

cudaError_t launch_gemv_q8k(const Q8kArgs &a, int sm_count, cudaStream_t s)
{
    Q8kParams P;
    memset(&P, 0, sizeof(P));
    int64_t tot = 0;
    for (int i = 0; i < a.nmat; ++i) {
        P.w[i] = a.w[i];
        P.y[i] = a.y[i];
        tot += a.N[i];
        P.row_end[i] = tot;
    }
    for (int i = a.nmat; i < kMaxGroup; ++i)
        P.row_end[i] = INT64_MAX;
    P.nmat = a.nmat;
    P.N = tot;
    P.NB = int(a.K / 256);
    P.row_bytes = (a.K / 256) * 144;
    P.xq = a.xq;
    P.x = a.x;
    // lanes per row: NB when it divides 32 (several rows per warp), else 32
    int lshift = 5;
    for (int l = 0; l <= 5; ++l)
        if ((1 << l) == P.NB)
            lshift = l;
    if (const char *e = getenv("QMM_Q8K_LSHIFT"))  // tuning override: log2(lanes per row)
        lshift = std::min(5, std::max(0, atoi(e)));
    P.lshift = lshift;
    const int64_t R = 32 >> lshift;
    P.n_groups = (tot + R - 1) / R;
    const size_t smem = q8k_smem(a.K);
    const auto kern = a.x ? gemv_q8k_kernel<true> : gemv_q8k_kernel<false>;
    cudaError_t e = func_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess)
        return e;
    const int64_t want = (P.n_groups + kWarps - 1) / kWarps;
    int64_t cap = int64_t(sm_count) * 2;
    if (const char *e = getenv("QMM_Q8K_CTAS"))  // tuning override: grid cap
        cap = std::max<int64_t>(1, atoll(e));
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, cap));
    return launch_pdl(kern, dim3(unsigned(grid)), dim3(32 * kWarps), smem, s, P);
}

} // namespace qmm
