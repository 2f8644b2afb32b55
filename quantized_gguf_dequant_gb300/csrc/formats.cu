// formats.cu -- decode GEMV and block decode for the further GGUF block
// formats (Q5_K, Q6_K, IQ4_NL; layouts in formats.cuh).
//
// The operation is the one of the other paths ("Building a Rust Inference
// Engine That Matches Llama.cpp", "Where the wins came from": the weights are
// decoded inline in the dot product, never expanded into a buffer), for the
// K-quants and IQ4_NL that "Frink Inference: the Rust alternative to
// llama.cpp" names ("Where Frink is already better than llama.cpp": the
// K-quants written byte-identically; "Where llama.cpp is still ahead":
// IQ4_NL).
//
// GEMV: one warp per output row; lane l decodes the row's 32-weight groups
// l, l+32, ... in registers and multiplies each by the M activation rows
// (M <= 16), accumulating in fp32; the lanes are then added by a fixed
// shuffle tree, so results are bitwise repeatable.  A plain design that reads
// bytes: it takes what the fast kernel of formats_fast.cu does not (Q8_0 and
// IQ4_NL rows whose K is not a multiple of 256, activations that do not fit
// shared memory) and is kept as the simple second implementation.
#include "formats.cuh"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kFmtWarps = 8;

template <int F, int MR>
__global__ void __launch_bounds__(kFmtWarps * 32) gemv_fmt_kernel(
    const uint8_t *__restrict__ w, int64_t N, int64_t K, int64_t row_bytes,
    const float *__restrict__ X, int M, int64_t ldx, float *__restrict__ Y, int64_t ldy)
{
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = int64_t(blockIdx.x) * kFmtWarps + warp;
    if (r >= N)
        return;
    const uint8_t *row = w + r * row_bytes;
    const int64_t groups = K / 32;
    float acc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m)
        acc[m] = 0.f;
    for (int64_t g = lane; g < groups; g += 32) {
        float v[32];
        fmt::decode_group<F>(row, g, v);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            if (m < M) {
                const float *x = X + int64_t(m) * ldx + g * 32;
                float s = 0.f;
#pragma unroll
                for (int l = 0; l < 32; ++l)
                    s = fmaf(v[l], __ldg(x + l), s);
                acc[m] += s;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        float a = acc[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0 && m < M)
            Y[int64_t(m) * ldy + r] = a;
    }
}

template <int F, bool BF16>
__global__ void dequant_fmt_kernel(const uint8_t *__restrict__ w, int64_t K, int64_t row_bytes,
                                   int64_t row0, int64_t nrows, float *__restrict__ of,
                                   __nv_bfloat16 *__restrict__ ob)
{
    const int64_t groups = K / 32;
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= nrows * groups)
        return;
    const int64_t r = gid / groups, g = gid % groups;
    float v[32];
    fmt::decode_group<F>(w + (row0 + r) * row_bytes, g, v);
    const int64_t o = r * K + g * 32;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        if (BF16)
            ob[o + l] = __float2bfloat16_rn(v[l]);
        else
            of[o + l] = v[l];
    }
}

template <int F>
cudaError_t launch_gemv_fmt_t(const Matrix &m, const float *X, int M, int64_t ldx, float *Y,
                              int64_t ldy, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((m.N + kFmtWarps - 1) / kFmtWarps));
    cfg.blockDim = dim3(kFmtWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    if (M == 1)
        return counted(cudaLaunchKernelEx(&cfg, gemv_fmt_kernel<F, 1>, m.w, m.N, m.K, m.row_bytes,
                                          X, M, ldx, Y, ldy));
    return counted(cudaLaunchKernelEx(&cfg, gemv_fmt_kernel<F, 16>, m.w, m.N, m.K, m.row_bytes, X,
                                      M, ldx, Y, ldy));
}

template <int F>
cudaError_t launch_dequant_fmt_t(const Matrix &m, int64_t row0, int64_t nrows, float *of,
                                 __nv_bfloat16 *ob, cudaStream_t s)
{
    const int64_t total = nrows * (m.K / 32);
    const int threads = 256;
    const unsigned blocks = unsigned((total + threads - 1) / threads);
    if (ob)
        dequant_fmt_kernel<F, true><<<blocks, threads, 0, s>>>(m.w, m.K, m.row_bytes, row0, nrows,
                                                               nullptr, ob);
    else
        dequant_fmt_kernel<F, false><<<blocks, threads, 0, s>>>(m.w, m.K, m.row_bytes, row0, nrows,
                                                                of, nullptr);
    return counted(cudaGetLastError());
}

} // namespace

bool is_extra_format(int f)
{
    return f == fmt::kQ5K || f == fmt::kQ6K || f == fmt::kIQ4NL;
}

bool uses_fmt_kernels(const Matrix &m)
{
    return is_extra_format(m.fmt) || (m.fmt == fmt::kQ80 && m.K % 256 != 0);
}

cudaError_t launch_gemv_fmt(const Matrix &m, const float *X, int M, int64_t ldx, float *Y,
                            int64_t ldy, cudaStream_t s)
{
    switch (m.fmt) {
    case fmt::kQ5K: return launch_gemv_fmt_t<fmt::kQ5K>(m, X, M, ldx, Y, ldy, s);
    case fmt::kQ6K: return launch_gemv_fmt_t<fmt::kQ6K>(m, X, M, ldx, Y, ldy, s);
    case fmt::kQ80: return launch_gemv_fmt_t<fmt::kQ80>(m, X, M, ldx, Y, ldy, s);
    default: return launch_gemv_fmt_t<fmt::kIQ4NL>(m, X, M, ldx, Y, ldy, s);
    }
}

cudaError_t launch_dequant_fmt(const Matrix &m, int64_t row0, int64_t nrows, float *out_f32,
                               uint16_t *out_bf16, cudaStream_t s)
{
    __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(out_bf16);
    switch (m.fmt) {
    case fmt::kQ5K: return launch_dequant_fmt_t<fmt::kQ5K>(m, row0, nrows, out_f32, ob, s);
    case fmt::kQ6K: return launch_dequant_fmt_t<fmt::kQ6K>(m, row0, nrows, out_f32, ob, s);
    case fmt::kQ80: return launch_dequant_fmt_t<fmt::kQ80>(m, row0, nrows, out_f32, ob, s);
    default: return launch_dequant_fmt_t<fmt::kIQ4NL>(m, row0, nrows, out_f32, ob, s);
    }
}

} // namespace qmm
