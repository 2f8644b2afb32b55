// qmm_api.cu -- the C ABI: argument checks that refuse by name, handle and
// workspace management, plan selection and launches.  Every check happens on
// the host before anything is launched; a refused call launches nothing.
//
// Refusal convention: "Frink Inference: the Rust alternative to llama.cpp",
// section "The goal, stated once" -- load, or refuse with a sentence naming
// exactly what is missing; never compute something else.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "qmm_internal.h"

using qmm::Matrix;

namespace {

thread_local std::string g_err;

qmm_status fail(qmm_status code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

qmm_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(QMM_ERR_CUDA, "%s: CUDA error %d (%s): %s", what, int(e), cudaGetErrorName(e),
                cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmm_status check_handle(qmm_t h, const char *fn)
{
    if (!h)
        return fail(QMM_ERR_NULL, "%s: the matrix handle is NULL", fn);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    if (dev != reinterpret_cast<Matrix *>(h)->device)
        return fail(QMM_ERR_CUDA,
                    "%s: the handle was created on device %d but device %d is current", fn,
                    reinterpret_cast<Matrix *>(h)->device, dev);
    return QMM_OK;
}

int env_int(const char *name)
{
    const char *v = getenv(name);
    return v ? atoi(v) : 0;
}

constexpr size_t kMaxSmem = 227 * 1024;

// Q4_K on the tensor cores for M activation rows (1..4) when the activations
// of this K fit in shared memory (with the largest CTA shape).  For a single
// activation row and a very long K the fp32 kernel is faster (the tensor-core
// kernel re-lays all of x out in every CTA first).  QMM_Q4K_PATH = "simt" or
// "tc" forces a path.
bool tc_fits(const Matrix &m0, int M)
{
    const char *path = getenv("QMM_Q4K_PATH");
    if (path && strcmp(path, "simt") == 0)
        return false;
    if (!m0.has_tmap || M < 1 || M > 4 || qmm::gemv_tc_smem(m0.K, M, 3, 16) > kMaxSmem)
        return false;
    if (path && strcmp(path, "tc") == 0)
        return true;
    return !(M == 1 && m0.K > 8192);
}

qmm_status do_gemv_tc(const qmm_t *hs, int n, const float *x, int64_t ldx, int M, float *const *ys,
                      int64_t ldy, cudaStream_t s, const char *fn)
{
    const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
    qmm::TcArgs a;
    memset(&a, 0, sizeof(a));
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
        a.tmap[i] = mi.tmap;
        a.rows[i] = mi.N;
        a.y[i] = ys[i];
        tiles += (mi.N + 15) / 16;
    }
    if (size_t(tiles) > m0.tc_tickets_n)
        return fail(QMM_ERR_NOMEM, "%s: %lld row tiles exceed handle 0's ticket array (%zu)", fn,
                    (long long)tiles, m0.tc_tickets_n);
    a.nmat = n;
    a.K = m0.K;
    a.M = M;
    a.ldx = ldx;
    a.ldy = ldy;
    a.x = x;
    a.ws = m0.tc_ws;
    a.tickets = m0.tc_tickets;
    a.status = m0.status;
    cudaError_t e = qmm::launch_gemv_tc(a, m0.sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
    return QMM_OK;
}

qmm_status do_gemv(const qmm_t *hs, int n, const float *x, float *const *ys, cudaStream_t s,
                   const char *fn)
{
    const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
    if (m0.fmt == QMM_Q4_K && tc_fits(m0, 1))
        return do_gemv_tc(hs, n, x, m0.K, 1, ys, 0, s, fn);
    qmm::GemvArgs a;
    memset(&a, 0, sizeof(a));
    a.fmt = m0.fmt;
    a.nmat = n;
    a.K = m0.K;
    a.row_bytes = m0.row_bytes;
    a.x = x;
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
        a.w[i] = mi.w;
        a.y[i] = ys[i];
        total += mi.N;
        a.row_end[i] = total;
    }
    for (int i = n; i < qmm::kMaxGroup; ++i)
        a.row_end[i] = total;
    a.N = total;
    a.status = m0.status;
    qmm::GemvPlan p = qmm::plan_gemv(m0.fmt, total, m0.K, m0.sm_count, env_int("QMM_SPLITK"));
    if (p.ksplit > 1 && (qmm::gemv_workspace_floats(p, total) > m0.ws_floats ||
                         size_t(p.row_slices) > m0.n_tickets)) {
        qmm::GemvPlan p1 = qmm::plan_gemv(m0.fmt, total, m0.K, m0.sm_count, 1);
        if (p1.kchunks > 256)
            return fail(QMM_ERR_NOMEM,
                        "%s: split-K over %lld rows needs a larger workspace than handle 0 holds",
                        fn, (long long)total);
        p = p1;
    }
    a.ws = m0.ws;
    a.tickets = m0.tickets;
    cudaError_t e = qmm::launch_gemv(p, a, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
    return QMM_OK;
}

} // namespace

namespace qmm {

qmm_status noalloc_fail(qmm_status code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

qmm_status noalloc_check(int fmt, int64_t N, int64_t K, const void *w, const float *x,
                         const float *y)
{
    g_err.clear();
    if (!w || !x || !y)
        return fail(QMM_ERR_NULL, "qmm_gemv_noalloc: %s is NULL", !w ? "the weight pointer"
                                                                 : (!x ? "x" : "y"));
    if (fmt != QMM_Q4_K && fmt != QMM_Q8_0)
        return fail(QMM_ERR_FORMAT,
                    "qmm_gemv_noalloc: format %d is not supported (Q4_K = 12 and Q8_0 = 8 are)",
                    fmt);
    if (N < 1)
        return fail(QMM_ERR_SHAPE, "qmm_gemv_noalloc: N = %lld rows; at least one row is needed",
                    (long long)N);
    if (K < 256 || K % 256 != 0 || K > (int64_t(1) << 20))
        return fail(QMM_ERR_SHAPE,
                    "qmm_gemv_noalloc: K = %lld is not a multiple of 256 in [256, 1048576]",
                    (long long)K);
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4))
        return fail(QMM_ERR_ALIGN, "qmm_gemv_noalloc: the weights and x must be 16-byte aligned "
                                   "and y 4-byte aligned");
    return QMM_OK;
}

} // namespace qmm

extern "C" {

const char *qmm_last_error(void) { return g_err.c_str(); }

int32_t qmm_version(void) { return 100; }

qmm_status qmm_create(qmm_format fmt, int64_t N, int64_t K, const void *w_dev, qmm_t *out)
{
    g_err.clear();
    if (!out)
        return fail(QMM_ERR_NULL, "qmm_create: the output handle pointer is NULL");
    *out = nullptr;
    if (!w_dev)
        return fail(QMM_ERR_NULL, "qmm_create: the weight pointer is NULL");
    if (fmt != QMM_Q4_K && fmt != QMM_Q8_0)
        return fail(QMM_ERR_FORMAT,
                    "qmm_create: format %d is not supported (Q4_K = 12 and Q8_0 = 8 are)", int(fmt));
    if (N < 1)
        return fail(QMM_ERR_SHAPE, "qmm_create: N = %lld rows; at least one row is needed",
                    (long long)N);
    if (K < 256 || K % 256 != 0)
        return fail(QMM_ERR_SHAPE,
                    fmt == QMM_Q4_K
                        ? "qmm_create: K = %lld is not a positive multiple of 256 (a Q4_K "
                          "super-block holds 256 weights)"
                        : "qmm_create: K = %lld is not a positive multiple of 256 (Q8_0 rows must "
                          "be 16-byte multiples here, which needs K %% 256 == 0)",
                    (long long)K);
    if (K > (int64_t(1) << 20))
        return fail(QMM_ERR_SHAPE, "qmm_create: K = %lld exceeds the supported maximum 1048576",
                    (long long)K);
    if (!aligned(w_dev, 16))
        return fail(QMM_ERR_ALIGN, "qmm_create: the weight pointer is not 16-byte aligned");
    Matrix *m = new Matrix;
    m->fmt = fmt;
    m->N = N;
    m->K = K;
    m->row_bytes = qmm::row_bytes_of(fmt, K);
    m->w = static_cast<const uint8_t *>(w_dev);
    cudaError_t e = cudaGetDevice(&m->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&m->sm_count, cudaDevAttrMultiProcessorCount, m->device);
    if (e != cudaSuccess) {
        delete m;
        return cuda_fail(e, "qmm_create");
    }
    m->ws_floats = size_t(8) * size_t(N) + 1024;
    m->n_tickets = size_t(m->sm_count) * 4;
    if (fmt == QMM_Q4_K) {
        if (qmm::make_q4k_tensor_map(m->tmap, w_dev, N, m->row_bytes) != 0) {
            delete m;
            return fail(QMM_ERR_CUDA, "qmm_create: the TMA tensor map for the weight rows could "
                                      "not be encoded (driver entry point or arguments refused)");
        }
        m->has_tmap = true;
        m->tc_ws_floats = qmm::gemv_tc_ws_floats(m->sm_count);
        m->tc_tickets_n = size_t(N > 32768 ? N : 32768) / 16 + 64;
    }
    void *p = nullptr;
    const size_t bytes = m->ws_floats * 4 + m->n_tickets * 4 + 256 + m->tc_ws_floats * 4 +
                         m->tc_tickets_n * 4;
    e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) {
        delete m;
        return fail(QMM_ERR_NOMEM, "qmm_create: could not allocate the %zu-byte workspace (%s)",
                    bytes, cudaGetErrorString(e));
    }
    e = cudaMemset(p, 0, bytes);
    if (e != cudaSuccess) {
        cudaFree(p);
        delete m;
        return cuda_fail(e, "qmm_create");
    }
    m->ws = static_cast<float *>(p);
    m->tickets = reinterpret_cast<unsigned *>(m->ws + m->ws_floats);
    m->status = m->tickets + m->n_tickets;
    m->tc_ws = reinterpret_cast<float *>(m->status + 64);
    m->tc_tickets = reinterpret_cast<unsigned *>(m->tc_ws + m->tc_ws_floats);
    *out = reinterpret_cast<qmm_t>(m);
    return QMM_OK;
}

qmm_status qmm_destroy(qmm_t h)
{
    g_err.clear();
    if (!h)
        return fail(QMM_ERR_NULL, "qmm_destroy: the matrix handle is NULL");
    Matrix *m = reinterpret_cast<Matrix *>(h);
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(m->device);
    cudaDeviceSynchronize();
    if (m->ws)
        cudaFree(m->ws);
    if (m->moe_ws)
        cudaFree(m->moe_ws);
    if (prev >= 0)
        cudaSetDevice(prev);
    delete m;
    return QMM_OK;
}

qmm_status qmm_gemv(qmm_t h, const float *x, float *y, qmm_stream stream)
{
    g_err.clear();
    qmm_status st = check_handle(h, "qmm_gemv");
    if (st != QMM_OK)
        return st;
    if (!x || !y)
        return fail(QMM_ERR_NULL, "qmm_gemv: %s is NULL", !x ? "x" : "y");
    if (!aligned(x, 16))
        return fail(QMM_ERR_ALIGN, "qmm_gemv: x is not 16-byte aligned");
    if (!aligned(y, 4))
        return fail(QMM_ERR_ALIGN, "qmm_gemv: y is not 4-byte aligned");
    float *ys[1] = {y};
    return do_gemv(&h, 1, x, ys, static_cast<cudaStream_t>(stream), "qmm_gemv");
}

qmm_status qmm_gemv_group(const qmm_t *hs, int32_t n, const float *x, float *const *ys,
                          qmm_stream stream)
{
    g_err.clear();
    if (!hs || !ys)
        return fail(QMM_ERR_NULL, "qmm_gemv_group: the %s array is NULL", !hs ? "handle" : "output");
    if (n < 1 || n > qmm::kMaxGroup)
        return fail(QMM_ERR_SHAPE, "qmm_gemv_group: n = %d; between 1 and %d matrices are supported",
                    int(n), qmm::kMaxGroup);
    for (int i = 0; i < n; ++i) {
        qmm_status st = check_handle(hs[i], "qmm_gemv_group");
        if (st != QMM_OK)
            return st;
        if (!ys[i])
            return fail(QMM_ERR_NULL, "qmm_gemv_group: output %d is NULL", i);
        if (!aligned(ys[i], 4))
            return fail(QMM_ERR_ALIGN, "qmm_gemv_group: output %d is not 4-byte aligned", i);
        const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
        const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
        if (mi.fmt != m0.fmt || mi.K != m0.K)
            return fail(QMM_ERR_SHAPE,
                        "qmm_gemv_group: matrix %d (format %d, K %lld) differs from matrix 0 "
                        "(format %d, K %lld); a group shares one format and one K",
                        i, mi.fmt, (long long)mi.K, m0.fmt, (long long)m0.K);
    }
    if (!x)
        return fail(QMM_ERR_NULL, "qmm_gemv_group: x is NULL");
    if (!aligned(x, 16))
        return fail(QMM_ERR_ALIGN, "qmm_gemv_group: x is not 16-byte aligned");
    return do_gemv(hs, n, x, ys, static_cast<cudaStream_t>(stream), "qmm_gemv_group");
}

qmm_status qmm_gemv_batched(qmm_t h, const float *X, int64_t M, int64_t ldx, float *Y,
                            int64_t ldy, qmm_stream stream)
{
    g_err.clear();
    qmm_status st = check_handle(h, "qmm_gemv_batched");
    if (st != QMM_OK)
        return st;
    const Matrix &m = *reinterpret_cast<const Matrix *>(h);
    if (!X || !Y)
        return fail(QMM_ERR_NULL, "qmm_gemv_batched: %s is NULL", !X ? "X" : "Y");
    if (M < 1 || M > 16)
        return fail(QMM_ERR_SHAPE, "qmm_gemv_batched: M = %lld; 1 <= M <= 16 is supported",
                    (long long)M);
    if (ldx < m.K || ldy < m.N)
        return fail(QMM_ERR_SHAPE, "qmm_gemv_batched: ldx = %lld < K = %lld or ldy = %lld < N = %lld",
                    (long long)ldx, (long long)m.K, (long long)ldy, (long long)m.N);
    if (ldx % 4 || !aligned(X, 16))
        return fail(QMM_ERR_ALIGN, "qmm_gemv_batched: X rows must start 16-byte aligned "
                                   "(X aligned and ldx a multiple of 4)");
    if (!aligned(Y, 4))
        return fail(QMM_ERR_ALIGN, "qmm_gemv_batched: Y is not 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Up to four activation rows share one pass over the weights; larger
    // batches take ceil(M/4) passes.
    for (int64_t m0 = 0; m0 < M;) {
        int mc = int(M - m0 < 4 ? M - m0 : 4);
        while (mc > 1 && !tc_fits(m, mc))
            --mc;
        float *yrow = Y + m0 * ldy;
        if (m.fmt == QMM_Q4_K && tc_fits(m, mc)) {
            st = do_gemv_tc(&h, 1, X + m0 * ldx, ldx, mc, &yrow, ldy, s, "qmm_gemv_batched");
        } else {
            mc = 1;
            st = do_gemv(&h, 1, X + m0 * ldx, &yrow, s, "qmm_gemv_batched");
        }
        if (st != QMM_OK)
            return st;
        m0 += mc;
    }
    return QMM_OK;
}

qmm_status qmm_moe_gemv(qmm_t h, int32_t n_experts, const int32_t *expert_ids, int32_t T,
                        int32_t top_k, const float *X, int32_t x_per_slot,
                        const float *route_w, float *Y, qmm_stream stream)
{
    g_err.clear();
    (void)h; (void)n_experts; (void)expert_ids; (void)T; (void)top_k; (void)X;
    (void)x_per_slot; (void)route_w; (void)Y; (void)stream;
    return fail(QMM_ERR_UNSUPPORTED, "qmm_moe_gemv: not implemented in this build");
}

qmm_status qmm_swiglu(const float *g, const float *u, float *hh, int64_t n, qmm_stream stream)
{
    g_err.clear();
    (void)g; (void)u; (void)hh; (void)n; (void)stream;
    return fail(QMM_ERR_UNSUPPORTED, "qmm_swiglu: not implemented in this build");
}

qmm_status qmm_moe_ffn(qmm_t hg, qmm_t hu, qmm_t hd, int32_t n_experts,
                       const int32_t *expert_ids, int32_t T, int32_t top_k, const float *X,
                       const float *route_w, float *Y, qmm_stream stream)
{
    g_err.clear();
    (void)hg; (void)hu; (void)hd; (void)n_experts; (void)expert_ids; (void)T; (void)top_k;
    (void)X; (void)route_w; (void)Y; (void)stream;
    return fail(QMM_ERR_UNSUPPORTED, "qmm_moe_ffn: not implemented in this build");
}

qmm_status qmm_gemm(qmm_t h, const uint16_t *X_bf16, int64_t M, float *Y, qmm_stream stream)
{
    g_err.clear();
    (void)h; (void)X_bf16; (void)M; (void)Y; (void)stream;
    return fail(QMM_ERR_UNSUPPORTED, "qmm_gemm: not implemented in this build");
}

static qmm_status dequant_common(qmm_t h, int64_t row0, int64_t nrows, float *of, uint16_t *ob,
                                 qmm_stream stream, const char *fn)
{
    g_err.clear();
    qmm_status st = check_handle(h, fn);
    if (st != QMM_OK)
        return st;
    const Matrix &m = *reinterpret_cast<const Matrix *>(h);
    if (!of && !ob)
        return fail(QMM_ERR_NULL, "%s: the output pointer is NULL", fn);
    if (row0 < 0 || nrows < 0 || row0 + nrows > m.N)
        return fail(QMM_ERR_SHAPE, "%s: rows %lld..%lld are outside the matrix's %lld rows", fn,
                    (long long)row0, (long long)(row0 + nrows), (long long)m.N);
    if (of && !aligned(of, 16))
        return fail(QMM_ERR_ALIGN, "%s: the output is not 16-byte aligned", fn);
    if (ob && !aligned(ob, 2))
        return fail(QMM_ERR_ALIGN, "%s: the output is not 2-byte aligned", fn);
    if (nrows == 0)
        return QMM_OK;
    cudaError_t e = qmm::launch_dequant(m, row0, nrows, of, ob, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(h)->last_stream = static_cast<cudaStream_t>(stream);
    return QMM_OK;
}

qmm_status qmm_dequantize(qmm_t h, int64_t row0, int64_t nrows, float *out, qmm_stream stream)
{
    return dequant_common(h, row0, nrows, out, nullptr, stream, "qmm_dequantize");
}

qmm_status qmm_dequantize_bf16(qmm_t h, int64_t row0, int64_t nrows, uint16_t *out,
                               qmm_stream stream)
{
    return dequant_common(h, row0, nrows, nullptr, out, stream, "qmm_dequantize_bf16");
}

qmm_status qmm_get_status(qmm_t h)
{
    g_err.clear();
    qmm_status st = check_handle(h, "qmm_get_status");
    if (st != QMM_OK)
        return st;
    Matrix *m = reinterpret_cast<Matrix *>(h);
    cudaError_t e = cudaStreamSynchronize(m->last_stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "qmm_get_status");
    unsigned word = 0;
    e = cudaMemcpy(&word, m->status, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        e = cudaMemset(m->status, 0, 4);
    if (e != cudaSuccess)
        return cuda_fail(e, "qmm_get_status");
    if (word & qmm::kStatusTimeoutBit)
        return fail(QMM_ERR_TIMEOUT, "qmm_get_status: a device-side pipeline wait gave up");
    if (word & qmm::kStatusBadExpertBit)
        return fail(QMM_ERR_EXPERT,
                    "qmm_get_status: an expert id was outside [0, n_experts); its slot was left 0");
    return QMM_OK;
}

} // extern "C"
