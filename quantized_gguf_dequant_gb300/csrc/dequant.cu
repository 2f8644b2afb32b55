// dequant.cu -- decode rows of a GGUF matrix to fp32 (or bf16) in global
// memory.  This is the inspection / test path (the products never
// materialise weights); it exposes exactly the per-weight values the fused
// kernels use, so they can be compared bit for bit with the oracle.
//
// Q4_K: w = d*sc*q - dmin*m.  d*sc and dmin*m are exact in fp32 (11+6 and
// 11+6 significant bits), so fmaf(d*sc, q, -(dmin*m)) rounds the exact weight
// once: the result is RN_fp32(w).  Q8_0: d*q (11+8 bits) is exact.
// bf16 output: round-to-nearest-even of that fp32 value.
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

// One thread decodes 32 consecutive weights (one Q4_K sub-block or one Q8_0
// block) of one row.
template <int FMT, bool BF16>
__global__ void dequant_kernel(const uint8_t *__restrict__ w, int64_t K, int64_t row_bytes,
                               int64_t row0, int64_t nrows, float *__restrict__ of,
                               __nv_bfloat16 *__restrict__ ob)
{
    const int64_t groups = K / 32;
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= nrows * groups)
        return;
    const int64_t r = gid / groups;
    const int64_t gi = gid % groups;  // 32-weight group within the row
    const uint8_t *row = w + (row0 + r) * row_bytes;
    float v[32];
    if (FMT == QMM_Q4_K) {
        const uint8_t *blk = row + (gi / 8) * 144;
        const int j = int(gi % 8);  // sub-block
        const uint8_t *sc12 = blk + 4;
        int sc, m;
        if (j < 4) {
            sc = sc12[j] & 63;
            m = sc12[j + 4] & 63;
        } else {
            sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
            m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
        }
        const float d = __half2float(*reinterpret_cast<const __half *>(blk));
        const float dmin = __half2float(*reinterpret_cast<const __half *>(blk + 2));
        const float a = d * float(sc);
        const float b = dmin * float(m);
        const uint8_t *qs = blk + 16 + 32 * (j / 2);
        const int shift = (j & 1) ? 4 : 0;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = fmaf(a, float((qs[i] >> shift) & 15), -b);
    } else {
        const uint8_t *blk = row + gi * 34;
        const float d = __half2float(__ushort_as_half(uint16_t(blk[0] | (blk[1] << 8))));
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = d * float(int8_t(blk[2 + i]));
    }
    const int64_t o = r * K + gi * 32;
    if (BF16) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            ob[o + i] = __float2bfloat16_rn(v[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(of + o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
}

} // namespace

cudaError_t launch_dequant(const Matrix &m, int64_t row0, int64_t nrows, float *out_f32,
                           uint16_t *out_bf16, cudaStream_t s)
{
    if (uses_fmt_kernels(m))
        return launch_dequant_fmt(m, row0, nrows, out_f32, out_bf16, s);
    const int64_t total = nrows * (m.K / 32);
    const int threads = 256;
    const unsigned blocks = unsigned((total + threads - 1) / threads);
    __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(out_bf16);
    if (m.fmt == QMM_Q4_K) {
        if (out_bf16)
            dequant_kernel<QMM_Q4_K, true><<<blocks, threads, 0, s>>>(m.w, m.K, m.row_bytes, row0,
                                                                      nrows, nullptr, ob);
        else
            dequant_kernel<QMM_Q4_K, false><<<blocks, threads, 0, s>>>(m.w, m.K, m.row_bytes, row0,
                                                                       nrows, out_f32, nullptr);
    } else {
        if (out_bf16)
            dequant_kernel<QMM_Q8_0, true><<<blocks, threads, 0, s>>>(m.w, m.K, m.row_bytes, row0,
                                                                      nrows, nullptr, ob);
        else
            dequant_kernel<QMM_Q8_0, false><<<blocks, threads, 0, s>>>(m.w, m.K, m.row_bytes, row0,
                                                                       nrows, out_f32, nullptr);
    }
    return counted(cudaGetLastError());
}

} // namespace qmm
