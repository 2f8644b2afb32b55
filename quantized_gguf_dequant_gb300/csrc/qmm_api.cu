// qmm_api.cu -- the C ABI: argument checks that refuse by name, handle and
// workspace management, plan selection and launches.  Every check happens on
// the host before anything is launched; a refused call launches nothing.
//
// Refusal convention: "Frink Inference: the Rust alternative to llama.cpp",
// section "The goal, stated once" -- load, or refuse with a sentence naming
// exactly what is missing; never compute something else.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <unordered_map>
#include <mutex>
#include <string>

#include <cuda.h>

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
    for (int i = 0; i < n; ++i) {
        const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
        a.tmap[i] = mi.tmap;
        a.rows[i] = mi.N;
        a.y[i] = ys[i];
    }
    a.nmat = n;
    a.K = m0.K;
    a.M = M;
    a.ldx = ldx;
    a.ldy = ldy;
    a.x = x;
    a.status = m0.status;
    cudaError_t e = qmm::launch_gemv_tc(a, m0.sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
    return QMM_OK;
}

// The one-pass batched tensor-core kernel (gemv_batched.cu) for M rows of one
// Q4_K matrix.  QMM_ERR_UNSUPPORTED (nothing launched) if the shape does not
// fit its shared memory.
qmm_status do_gemv_tcb(qmm_t h, const float *X, int64_t ldx, int M, float *Y, int64_t ldy,
                       cudaStream_t s, const char *fn)
{
    Matrix &mm = *reinterpret_cast<Matrix *>(h);
    const qmm::TcbPlan p = qmm::plan_tcb(mm.N, mm.K, M, mm.sm_count);
    if (p.S == 0)
        return QMM_ERR_UNSUPPORTED;
    const size_t need = p.ws_floats * 4;
    if (need > mm.tcb_ws_bytes) {
        cudaError_t e = cudaSuccess;
        if (mm.tcb_ws) {
            e = cudaDeviceSynchronize();
            if (e == cudaSuccess)
                e = cudaFree(mm.tcb_ws);
            mm.tcb_ws = nullptr;
            mm.tcb_ws_bytes = 0;
            if (e != cudaSuccess)
                return cuda_fail(e, fn);
        }
        void *ptr = nullptr;
        e = cudaMalloc(&ptr, need);
        if (e != cudaSuccess)
            return fail(QMM_ERR_NOMEM, "%s: could not allocate %zu bytes of K-slice scratch (%s)", fn,
                        need, cudaGetErrorString(e));
        mm.tcb_ws = ptr;
        mm.tcb_ws_bytes = need;
    }
    qmm::TcbArgs a;
    memset(&a, 0, sizeof(a));
    a.tmap = mm.tmap;
    a.x = X;
    a.y = Y;
    a.ws = p.S > 1 ? static_cast<float *>(mm.tcb_ws) : nullptr;
    if (p.tickets > mm.n_tickets)
        return fail(QMM_ERR_UNSUPPORTED, "%s: the K-sliced plan needs %zu row-group tickets, the "
                    "handle holds %zu", fn, p.tickets, mm.n_tickets);
    a.tickets = mm.tickets;
    a.status = mm.status;
    a.ldx = ldx;
    a.ldy = ldy;
    a.N = mm.N;
    a.K = mm.K;
    a.M = M;
    cudaError_t e = qmm::launch_gemv_tcb(a, p, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    mm.last_stream = s;
    return QMM_OK;
}

// The batched decode on tcgen05 (gemv_tc5.cu) for 2..16 rows of one Q4_K
// matrix: prepared activations, slice partials and tickets live in the
// handle's tc5 buffer (grown on demand: a synchronising allocation, so warm
// up before capturing a graph).
qmm_status do_gemv_tc5(qmm_t h, const float *X, int64_t ldx, int M, float *Y, int64_t ldy,
                       cudaStream_t s, const char *fn)
{
    Matrix &mm = *reinterpret_cast<Matrix *>(h);
    if (!mm.has_gemm_maps || mm.fmt != QMM_Q4_K || M < 2 || M > 16)
        return QMM_ERR_UNSUPPORTED;
    const qmm::Tc5Plan p = qmm::plan_tc5(mm.N, mm.K, M, mm.sm_count);
    const size_t prep = (p.prep_bytes + 255) & ~size_t(255);
    const size_t wsb = (p.ws_floats * 4 + 255) & ~size_t(255);
    const size_t need = prep + wsb + p.tickets * 4;
    if (need > mm.tc5_bytes) {
        cudaError_t e = cudaSuccess;
        if (mm.tc5_buf) {
            e = cudaDeviceSynchronize();
            if (e == cudaSuccess)
                e = cudaFree(mm.tc5_buf);
            mm.tc5_buf = nullptr;
            mm.tc5_bytes = 0;
            mm.tc5_nc = 0;
            if (e != cudaSuccess)
                return cuda_fail(e, fn);
        }
        void *ptr = nullptr;
        e = cudaMalloc(&ptr, need);
        if (e == cudaSuccess)
            e = cudaMemset(ptr, 0, need);  // the tickets start at zero
        if (e != cudaSuccess) {
            if (ptr)
                cudaFree(ptr);
            return fail(QMM_ERR_NOMEM, "%s: could not allocate %zu bytes of batched-decode scratch "
                        "(%s)", fn, need, cudaGetErrorString(e));
        }
        mm.tc5_buf = ptr;
        mm.tc5_bytes = need;
    }
    uint8_t *buf = static_cast<uint8_t *>(mm.tc5_buf);
    // The tickets sit at the end of the buffer, where every plan of this
    // handle finds them (zero between launches).
    unsigned *tickets = reinterpret_cast<unsigned *>(buf + mm.tc5_bytes) - p.tickets;
    if (reinterpret_cast<uint8_t *>(tickets) < buf + prep + wsb)
        return fail(QMM_ERR_NOMEM, "%s: batched-decode scratch too small", fn);
    if (mm.tc5_nc != p.nc) {
        if (qmm::encode_tmap_2d(mm.tc5_tmap_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, buf,
                                uint64_t(mm.K), uint64_t(p.nc), uint64_t(mm.K) * 2, 64u,
                                uint32_t(p.nc), CU_TENSOR_MAP_SWIZZLE_128B) != 0)
            return fail(QMM_ERR_CUDA, "%s: the tensor map of the prepared activations could not "
                                      "be encoded", fn);
        mm.tc5_nc = p.nc;
    }
    qmm::Tc5Args a;
    memset(&a, 0, sizeof(a));
    a.tmap_hdr = mm.tmap_hdr;
    a.tmap_nib = mm.tmap_nib;
    a.tmap_b = mm.tc5_tmap_b;
    a.prep = buf;
    a.ws = p.S > 1 ? reinterpret_cast<float *>(buf + prep) : nullptr;
    a.tickets = tickets;
    a.X = X;
    a.ldx = ldx;
    a.Y = Y;
    a.ldy = ldy;
    a.N = mm.N;
    a.K = mm.K;
    a.T = M;
    a.status = mm.status;
    cudaError_t e = qmm::launch_gemv_tc5(p, a, mm.sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    mm.last_stream = s;
    return QMM_OK;
}

// The one-row Q4_K / Q5_K decode kernel (gemv_m1.cu) for n matrices sharing x.
// QMM_ERR_UNSUPPORTED (nothing launched) when no plan fits its shared memory
// or the handle's workspace.  QMM_M1_S fixes the number of K slices.
qmm_status do_gemv_m1(const qmm_t *hs, int n, const float *x, float *const *ys, cudaStream_t s,
                      const char *fn, bool fuse = false)
{
    const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
    // fuse (gate, up): ys[0] = silu(gate x) * (up x), the pair's tiles interleaved
    if (fuse && (n != 2 || reinterpret_cast<const Matrix *>(hs[1])->N != m0.N))
        return QMM_ERR_UNSUPPORTED;
    const int min_ts = fuse ? 2 : 1;
    // units per warp and slot: 2 for the fused pairs (a warp takes a gate
    // tile's unit and its up tile's), else 1
    const int upw = fuse ? 2 : 1;
    qmm::M1Args a;
    memset(&a, 0, sizeof(a));
    int64_t T = 0;
    for (int i = 0; i < n; ++i) {
        const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
        if ((mi.fmt != QMM_Q4_K && mi.fmt != QMM_Q5_K && mi.fmt != QMM_Q6_K &&
             mi.fmt != QMM_IQ4_NL && mi.fmt != QMM_Q8_0) || mi.K % 256 != 0)
            return QMM_ERR_UNSUPPORTED;
        // Q6_K: TMA boxes of 8 super-blocks (1680 bytes) need K % 2048 == 0
        if (mi.fmt == QMM_Q6_K && mi.K % 2048 != 0)
            return QMM_ERR_UNSUPPORTED;
        a.rows[i] = mi.N;
        a.y[i] = ys[i];
        T += (mi.N + 15) / 16;
    }
    if (T * 16 > (int64_t(1) << 30))
        return QMM_ERR_UNSUPPORTED;
    const int64_t NB = m0.K / 256;
    // bytes of 256 weights: Q4_K / IQ4_NL 144, Q5_K 176, Q6_K 210, Q8_0 272
    const int sbb = m0.fmt == QMM_Q5_K   ? 176
                    : m0.fmt == QMM_Q6_K ? 210
                    : m0.fmt == QMM_Q8_0 ? 272
                                         : 144;
    qmm::M1Plan p = qmm::plan_m1(T, NB, m0.sm_count, 0, 0, sbb, min_ts, upw);
    // Fewer K slices when the handle's workspace or tickets are too small.
    for (int S = p.S; S >= 1 && (p.ws_floats > m0.ws_floats || p.tickets > m0.n_tickets); --S)
        if (NB % S == 0)
            p = qmm::plan_m1(T, NB, m0.sm_count, S, 0, sbb, min_ts, upw);
    if (p.nslot < 2 || p.ws_floats > m0.ws_floats || p.tickets > m0.n_tickets)
        return QMM_ERR_UNSUPPORTED;
    // Each matrix's column view with boxes of this plan's pass width (kept
    // in the handle; re-encoded when a plan asks for another width).
    for (int i = 0; i < n; ++i) {
        Matrix &mi = *reinterpret_cast<Matrix *>(hs[i]);
        if (mi.tmap3_ks != p.WS) {
            // Q6_K: a 2-D view of the rows as u64 words, boxes of 8
            // super-blocks (210 words) x 16 rows
            const int r = mi.fmt == QMM_Q6_K
                              ? qmm::encode_tmap_2d(mi.tmap3, CU_TENSOR_MAP_DATA_TYPE_UINT64, mi.w,
                                                    uint64_t(mi.row_bytes / 8), uint64_t(mi.N),
                                                    uint64_t(mi.row_bytes), 210u, 16u,
                                                    CU_TENSOR_MAP_SWIZZLE_NONE)
                              : qmm::make_column_map(mi.tmap3, mi.w, mi.N, mi.row_bytes, p.WS, sbb);
            if (r != 0)
                return QMM_ERR_UNSUPPORTED;
            mi.tmap3_ks = p.WS;
        }
        a.tmap[i] = mi.tmap3;
    }
    a.fmt = m0.fmt;
    a.nmat = n;
    a.x = x;
    a.fuse_swiglu = fuse ? 1 : 0;
    a.ws = m0.ws;
    a.tickets = m0.tickets;
    a.status = m0.status;
    cudaError_t e = qmm::launch_gemv_m1(a, p, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
    return QMM_OK;
}

// The staged fp32 GEMV (gemv.cu) for n matrices sharing x, with a given
// plan (its K-slice partials in handle 0's workspace).
qmm_status do_gemv_staged(const qmm_t *hs, int n, const float *x, float *const *ys,
                          const qmm::GemvPlan &p, cudaStream_t s, const char *fn)
{
    const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
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
    a.ws = m0.ws;
    a.tickets = m0.tickets;
    cudaError_t e = qmm::launch_gemv(p, a, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
    return QMM_OK;
}

// Weight bytes up to which a Q4_K GEMV (one row, a matrix or a group) takes
// the SIMT kernel instead of the decode kernel (QMM_Q4K_SMALL_BYTES; 0 by
// default).  Measured on the 1024 x 1024 matrix: the same 8.8 us for one
// call with L2 flushed, and in a CUDA graph of 512 distinct copies the
// decode kernel is faster (2.7 against 3.0 us per launch); eager calls of
// 1024 x 4096 favour the SIMT kernel (8.9 against 11.0 us).
int64_t q4k_small_bytes()
{
    const char *e = getenv("QMM_Q4K_SMALL_BYTES");
    return e ? int64_t(atoll(e)) : int64_t(0);
}

qmm_status do_gemv(const qmm_t *hs, int n, const float *x, float *const *ys, cudaStream_t s,
                   const char *fn)
{
    const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
    // Q4_K takes the SIMT kernel of formats_fast.cu only when asked
    // (QMM_Q4K_PATH=fmt) or when the group's weights are small enough that
    // the decode kernel's fixed set-up dominates (QMM_Q4K_SMALL_BYTES).
    bool simt_ok = m0.fmt != QMM_Q4_K;
    if (m0.fmt == QMM_Q4_K) {
        const char *qp = getenv("QMM_Q4K_PATH");
        int64_t bytes = 0;
        for (int i = 0; i < n; ++i)
            bytes += reinterpret_cast<const Matrix *>(hs[i])->N * m0.row_bytes;
        simt_ok = (qp && strcmp(qp, "fmt") == 0) || (!qp && bytes <= q4k_small_bytes());
    }
    // Q6_K takes the staged fp32 kernel where its 32-lane teams and 16-byte
    // bulk copies fit (measured on the Llama-3.1-8B shapes: 0.358 against
    // 0.406 ms for 4 layers on the SIMT kernel); Q5_K and IQ4_NL measured
    // faster on the SIMT kernel (0.266 / 0.287 against 0.334 / 0.364 ms).
    // QMM_FMT_PATH = staged, fast or plain picks the route for all three.
    const char *fp = getenv("QMM_FMT_PATH");
    // Q5_K, Q6_K, IQ4_NL and Q8_0: the tensor-core decode kernel of Q4_K with
    // the high bits added to the operands (IQ4_NL: the looked-up codes; Q8_0:
    // the bytes themselves) (QMM_FMT_PATH=staged, fast or plain keeps it off).
    if ((m0.fmt == QMM_Q5_K || m0.fmt == QMM_Q6_K || m0.fmt == QMM_IQ4_NL ||
         (m0.fmt == QMM_Q8_0 && m0.K % 256 == 0)) && !fp) {
        qmm_status st = do_gemv_m1(hs, n, x, ys, s, fn);
        if (st != QMM_ERR_UNSUPPORTED)
            return st;
    }
    const bool staged_pref = fp ? strcmp(fp, "staged") == 0 : m0.fmt == QMM_Q6_K;
    if (qmm::is_extra_format(m0.fmt) && m0.K % 256 == 0 && staged_pref) {
        int64_t total = 0;
        for (int i = 0; i < n; ++i)
            total += reinterpret_cast<const Matrix *>(hs[i])->N;
        qmm::GemvPlan p = qmm::plan_gemv(m0.fmt, total, m0.K, m0.sm_count, env_int("QMM_SPLITK"));
        if (qmm::gemv_plan_takes(m0.fmt, p, m0.row_bytes) &&
            qmm::gemv_workspace_floats(p, total) <= m0.ws_floats &&
            size_t(p.row_slices) <= m0.n_tickets)
            return do_gemv_staged(hs, n, x, ys, p, s, fn);
    }
    if (simt_ok && qmm::fmt_fast_rows(m0, 1) > 0) {
        const Matrix *ms[qmm::kMaxGroup];
        for (int i = 0; i < n; ++i)
            ms[i] = reinterpret_cast<const Matrix *>(hs[i]);
        cudaError_t e = qmm::launch_gemv_fmt_fast(ms, n, x, m0.K, 1, ys, 0, s);
        if (e != cudaSuccess)
            return cuda_fail(e, fn);
        reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
        return QMM_OK;
    }
    if (qmm::uses_fmt_kernels(m0)) {
        for (int i = 0; i < n; ++i) {
            const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
            cudaError_t e = qmm::launch_gemv_fmt(mi, x, 1, mi.K, ys[i], mi.N, s);
            if (e != cudaSuccess)
                return cuda_fail(e, fn);
        }
        reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
        return QMM_OK;
    }
    const char *qpath = getenv("QMM_Q4K_PATH");
    if (m0.fmt == QMM_Q4_K && !(qpath && (strcmp(qpath, "simt") == 0 || strcmp(qpath, "tc") == 0))) {
        qmm_status st = do_gemv_m1(hs, n, x, ys, s, fn);
        if (st != QMM_ERR_UNSUPPORTED)
            return st;
    }
    if (m0.fmt == QMM_Q4_K && tc_fits(m0, 1))
        return do_gemv_tc(hs, n, x, m0.K, 1, ys, 0, s, fn);
    // One Q4_K matrix whose x does not fit the decode kernel (K > 8192): the
    // K-sliced tensor-core kernel (measured faster than the fp32 kernel).
    if (m0.fmt == QMM_Q4_K && n == 1 && !(getenv("QMM_Q4K_PATH") &&
                                          strcmp(getenv("QMM_Q4K_PATH"), "simt") == 0)) {
        qmm_status st = do_gemv_tcb(hs[0], x, m0.K, 1, ys[0], m0.N, s, fn);
        if (st != QMM_ERR_UNSUPPORTED)
            return st;
    }
    int64_t total = 0;
    for (int i = 0; i < n; ++i)
        total += reinterpret_cast<const Matrix *>(hs[i])->N;
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
    return do_gemv_staged(hs, n, x, ys, p, s, fn);
}

// ------------------------------------------------------------------ experts

// Checks shared by the expert entry points, for one stacked handle.
qmm_status moe_check(const Matrix &m, int n_experts, const int32_t *ids, int T, int top_k,
                     const char *fn)
{
    if (m.fmt != QMM_Q4_K && !(m.fmt == QMM_Q8_0 && m.has_moe_map))
        return fail(QMM_ERR_UNSUPPORTED,
                    "%s: the expert GEMV is implemented for Q4_K weights and for Q8_0 weights "
                    "with K a multiple of 256 (this handle is format %d, K = %lld)", fn, m.fmt,
                    (long long)m.K);
    if (!ids)
        return fail(QMM_ERR_NULL, "%s: expert_ids is NULL", fn);
    if (n_experts < 1 || n_experts > qmm::kMoeMaxExperts)
        return fail(QMM_ERR_SHAPE, "%s: n_experts = %d; 1 <= n_experts <= %d is supported", fn,
                    n_experts, qmm::kMoeMaxExperts);
    if (m.N % n_experts != 0)
        return fail(QMM_ERR_SHAPE, "%s: the handle's %lld rows do not split into %d equal experts",
                    fn, (long long)m.N, n_experts);
    if (top_k < 1 || top_k > qmm::kMoeMaxTopK)
        return fail(QMM_ERR_SHAPE, "%s: top_k = %d; 1 <= top_k <= %d is supported", fn, top_k,
                    qmm::kMoeMaxTopK);
    if (T < 1 || int64_t(T) * top_k > qmm::kMoeMaxSlots)
        return fail(QMM_ERR_SHAPE, "%s: T = %d tokens x top_k = %d; 1 <= T*top_k <= %d is "
                    "supported", fn, T, top_k, qmm::kMoeMaxSlots);
    if (!aligned(ids, 4))
        return fail(QMM_ERR_ALIGN, "%s: expert_ids is not 4-byte aligned", fn);
    int nw, nslot;
    qmm::moe_expert_shape(m.K, nw, nslot);
    if (m.fmt == QMM_Q4_K && qmm::moe_expert_smem(m.K, nw, nslot, 0) > kMaxSmem)
        return fail(QMM_ERR_SHAPE, "%s: K = %lld is too long for the expert kernel's shared "
                    "memory (%zu bytes needed)", fn, (long long)m.K,
                    qmm::moe_expert_smem(m.K, nw, nslot, 0));
    return QMM_OK;
}

struct MoeScratch {
    qmm::MoeIndex ix;
    float *ys, *g, *u, *h;
};

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// The handle's expert scratch: the bucketing tables, ys_floats per-slot
// outputs and, for the FFN, three [S][d_ff] intermediates (ff_floats each).
// It grows when a call needs more; growing waits for the device first.
qmm_status moe_scratch(Matrix &m, int S, int E, size_t ys_floats, size_t ff_floats,
                       const char *fn, MoeScratch &out)
{
    const size_t o_groups = 0;
    const size_t o_slots = o_groups + round256(qmm::moe_max_groups(S, E) * sizeof(int4));
    const size_t o_ng = o_slots + round256(size_t(S) * sizeof(int));
    const size_t o_ys = o_ng + 256;
    const size_t o_g = o_ys + round256(ys_floats * 4);
    const size_t o_u = o_g + round256(ff_floats * 4);
    const size_t o_h = o_u + round256(ff_floats * 4);
    const size_t total = o_h + round256(ff_floats * 4);
    if (total > m.moe_ws_bytes) {
        cudaError_t e = cudaSuccess;
        if (m.moe_ws) {
            e = cudaDeviceSynchronize();
            if (e == cudaSuccess)
                e = cudaFree(m.moe_ws);
            m.moe_ws = nullptr;
            m.moe_ws_bytes = 0;
            if (e != cudaSuccess)
                return cuda_fail(e, fn);
        }
        void *p = nullptr;
        e = cudaMalloc(&p, total);
        if (e != cudaSuccess)
            return fail(QMM_ERR_NOMEM, "%s: could not allocate %zu bytes of expert scratch (%s)",
                        fn, total, cudaGetErrorString(e));
        m.moe_ws = p;
        m.moe_ws_bytes = total;
    }
    unsigned char *b = static_cast<unsigned char *>(m.moe_ws);
    out.ix.groups = reinterpret_cast<int4 *>(b + o_groups);
    out.ix.slots = reinterpret_cast<int *>(b + o_slots);
    out.ix.n_groups = reinterpret_cast<int *>(b + o_ng);
    out.ys = reinterpret_cast<float *>(b + o_ys);
    out.g = reinterpret_cast<float *>(b + o_g);
    out.u = reinterpret_cast<float *>(b + o_u);
    out.h = reinterpret_cast<float *>(b + o_h);
    return QMM_OK;
}

} // namespace

namespace qmm {

namespace {
std::atomic<int64_t> g_launches{0};
}

namespace {
// Function attributes already set, per (device, function): the shared-
// memory limit (threads = smem = 0 in the key), and resident blocks per SM
// (per threads and shared memory).
struct FuncKey {
    int dev;
    const void *func;
    int threads;
    size_t smem;
    bool operator==(const FuncKey &o) const
    {
        return dev == o.dev && func == o.func && threads == o.threads && smem == o.smem;
    }
};
struct FuncKeyHash {
    size_t operator()(const FuncKey &k) const
    {
        return std::hash<const void *>()(k.func) ^ (size_t(k.dev) << 48) ^ (size_t(k.threads) << 32) ^
               k.smem;
    }
};
std::mutex g_func_mu;
std::unordered_map<FuncKey, size_t, FuncKeyHash> g_func_smem;
std::unordered_map<FuncKey, int, FuncKeyHash> g_func_occ;
} // namespace

cudaError_t func_smem(const void *func, size_t bytes, bool max_carveout)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const FuncKey key{dev, func, 0, 0};
    std::lock_guard<std::mutex> lock(g_func_mu);
    auto it = g_func_smem.find(key);
    if (it != g_func_smem.end() && it->second >= bytes)
        return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess)
        g_func_smem[key] = bytes;
    return e;
}

cudaError_t func_occupancy(const void *func, int threads, size_t smem, int *per_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const FuncKey key{dev, func, threads, smem};
    std::lock_guard<std::mutex> lock(g_func_mu);
    auto it = g_func_occ.find(key);
    if (it != g_func_occ.end()) {
        *per_sm = it->second;
        return cudaSuccess;
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, func, threads, smem);
    if (e == cudaSuccess)
        g_func_occ[key] = *per_sm;
    return e;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

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
    const int64_t kb = fmt == QMM_Q8_0 ? 32 : 256;
    if (K < kb || K % kb != 0 || K > (int64_t(1) << 20))
        return fail(QMM_ERR_SHAPE,
                    "qmm_gemv_noalloc: K = %lld is not a multiple of %lld in [%lld, 1048576]",
                    (long long)K, (long long)kb, (long long)kb);
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4))
        return fail(QMM_ERR_ALIGN, "qmm_gemv_noalloc: the weights and x must be 16-byte aligned "
                                   "and y 4-byte aligned");
    return QMM_OK;
}

} // namespace qmm

extern "C" {

const char *qmm_last_error(void) { return g_err.c_str(); }

int32_t qmm_version(void) { return 100; }

int64_t qmm_launch_count(void) { return qmm::g_launches.load(std::memory_order_relaxed); }

qmm_status qmm_create(qmm_format fmt, int64_t N, int64_t K, const void *w_dev, qmm_t *out)
{
    g_err.clear();
    if (!out)
        return fail(QMM_ERR_NULL, "qmm_create: the output handle pointer is NULL");
    *out = nullptr;
    if (!w_dev)
        return fail(QMM_ERR_NULL, "qmm_create: the weight pointer is NULL");
    if (fmt != QMM_Q4_K && fmt != QMM_Q8_0 && !qmm::is_extra_format(fmt))
        return fail(QMM_ERR_FORMAT,
                    "qmm_create: format %d is not supported (Q4_K = 12, Q8_0 = 8, Q5_K = 13, "
                    "Q6_K = 14 and IQ4_NL = 20 are)", int(fmt));
    if (N < 1)
        return fail(QMM_ERR_SHAPE, "qmm_create: N = %lld rows; at least one row is needed",
                    (long long)N);
    const bool block32 = fmt == QMM_Q8_0 || fmt == QMM_IQ4_NL;
    if (block32 ? (K < 32 || K % 32 != 0) : (K < 256 || K % 256 != 0))
        return fail(QMM_ERR_SHAPE,
                    block32 ? "qmm_create: K = %lld is not a positive multiple of 32 (a block "
                              "holds 32 weights)"
                            : "qmm_create: K = %lld is not a positive multiple of 256 (a K-quant "
                              "super-block holds 256 weights)",
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
    // Row-group tickets of the split-K paths, and the item counters and
    // tickets of the one-row decode kernel (one per 16-row tile at most).
    m->n_tickets = size_t(m->sm_count) * 4 + size_t((N + 15) / 16) + 64;
    if (fmt == QMM_Q4_K) {
        if (qmm::make_q4k_tensor_map(m->tmap, w_dev, N, m->row_bytes) != 0) {
            delete m;
            return fail(QMM_ERR_CUDA, "qmm_create: the TMA tensor map for the weight rows could "
                                      "not be encoded (driver entry point or arguments refused)");
        }
        m->has_tmap = true;
        if (qmm::encode_tmap_2d(m->tmap_hdr, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_dev,
                                uint64_t(m->row_bytes), uint64_t(N), uint64_t(m->row_bytes), 16u,
                                256u, CU_TENSOR_MAP_SWIZZLE_NONE) != 0 ||
            qmm::encode_tmap_2d(m->tmap_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_dev,
                                uint64_t(m->row_bytes), uint64_t(N), uint64_t(m->row_bytes), 32u,
                                256u, CU_TENSOR_MAP_SWIZZLE_NONE) != 0) {
            delete m;
            return fail(QMM_ERR_CUDA, "qmm_create: the TMA tensor maps for the prefill GEMM "
                                      "could not be encoded");
        }
        m->has_gemm_maps = true;
    } else if (fmt == QMM_Q8_0 && K % 256 == 0) {
        // prefill GEMM: 80-byte windows over the rows (two 34-byte blocks
        // from the 16-byte boundary at or below them), 256 rows
        if (qmm::encode_tmap_2d(m->tmap_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_dev,
                                uint64_t(m->row_bytes), uint64_t(N), uint64_t(m->row_bytes), 80u,
                                256u, CU_TENSOR_MAP_SWIZZLE_NONE) != 0) {
            delete m;
            return fail(QMM_ERR_CUDA, "qmm_create: the TMA tensor map for the prefill GEMM "
                                      "could not be encoded");
        }
        m->has_gemm_maps = true;
        if (qmm::encode_moe_q8_map(m->tmap_moe, w_dev, N, m->row_bytes) != 0) {
            delete m;
            return fail(QMM_ERR_CUDA, "qmm_create: the TMA tensor map for the expert GEMV "
                                      "could not be encoded");
        }
        m->has_moe_map = true;
    }
    void *p = nullptr;
    const size_t bytes = m->ws_floats * 4 + m->n_tickets * 4 + 256;
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
    if (fmt == QMM_Q4_K) {
        // K-slice scratch of the one-pass tensor-core kernel for one
        // activation row (the M = 1 path when K is too long for the decode
        // kernel), so that qmm_gemv never allocates.
        const size_t need = qmm::plan_tcb(N, K, 1, m->sm_count).ws_floats * 4;
        if (need > 0) {
            e = cudaMalloc(&m->tcb_ws, need);
            if (e != cudaSuccess) {
                cudaFree(p);
                delete m;
                return fail(QMM_ERR_NOMEM, "qmm_create: could not allocate %zu bytes of K-slice "
                                           "scratch (%s)", need, cudaGetErrorString(e));
            }
            m->tcb_ws_bytes = need;
        }
    }
    m->tickets = reinterpret_cast<unsigned *>(m->ws + m->ws_floats);
    m->status = m->tickets + m->n_tickets;
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
    if (m->gemm_ws)
        cudaFree(m->gemm_ws);
    if (m->tcb_ws)
        cudaFree(m->tcb_ws);
    if (m->tc5_buf)
        cudaFree(m->tc5_buf);
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
    if (m.fmt != QMM_Q4_K && qmm::fmt_fast_rows(m, int(M)) > 0) {
        const Matrix *mp = &m;
        cudaError_t e = qmm::launch_gemv_fmt_fast(&mp, 1, X, ldx, int(M), &Y, ldy, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "qmm_gemv_batched");
        reinterpret_cast<Matrix *>(h)->last_stream = s;
        return QMM_OK;
    }
    if (qmm::uses_fmt_kernels(m)) {
        cudaError_t e = qmm::launch_gemv_fmt(m, X, int(M), ldx, Y, ldy, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "qmm_gemv_batched");
        reinterpret_cast<Matrix *>(h)->last_stream = s;
        return QMM_OK;
    }
    if (M == 1)  // one row: the decode GEMV itself
        return do_gemv(&h, 1, X, &Y, s, "qmm_gemv_batched");
    const char *bpath = getenv("QMM_BATCHED_PATH");
    const bool force_passes = bpath && strcmp(bpath, "passes") == 0;
    if (m.fmt == QMM_Q4_K && M >= 2 && !force_passes) {
        // All rows in one pass over the weights: the mma.sync kernel (the
        // default: measured faster at every Llama shape and M = 4..16), or
        // the tcgen05 kernel (QMM_BATCHED_PATH=tc5).
        if (bpath && strcmp(bpath, "tc5") == 0) {
            st = do_gemv_tc5(h, X, ldx, int(M), Y, ldy, s, "qmm_gemv_batched");
            if (st != QMM_ERR_UNSUPPORTED)
                return st;
        }
        st = do_gemv_tcb(h, X, ldx, int(M), Y, ldy, s, "qmm_gemv_batched");
        if (st != QMM_ERR_UNSUPPORTED)
            return st;
    }
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
                        const float *route_w, int32_t route_on_input, float *Y,
                        qmm_stream stream)
{
    g_err.clear();
    const char *fn = "qmm_moe_gemv";
    qmm_status st = check_handle(h, fn);
    if (st != QMM_OK)
        return st;
    Matrix *m = reinterpret_cast<Matrix *>(h);
    st = moe_check(*m, n_experts, expert_ids, T, top_k, fn);
    if (st != QMM_OK)
        return st;
    if (!X || !Y)
        return fail(QMM_ERR_NULL, "%s: %s is NULL", fn, !X ? "X" : "Y");
    if (x_per_slot != 0 && x_per_slot != 1)
        return fail(QMM_ERR_SHAPE, "%s: x_per_slot = %d; it must be 0 or 1", fn, x_per_slot);
    if (route_on_input != 0 && route_on_input != 1)
        return fail(QMM_ERR_SHAPE, "%s: route_on_input = %d; it must be 0 or 1", fn,
                    route_on_input);
    if (route_on_input && !route_w)
        return fail(QMM_ERR_NULL, "%s: route_on_input = 1 needs route_w", fn);
    if (!aligned(X, 16))
        return fail(QMM_ERR_ALIGN, "%s: X is not 16-byte aligned", fn);
    if (!aligned(Y, 4) || (route_w && !aligned(route_w, 4)))
        return fail(QMM_ERR_ALIGN, "%s: %s is not 4-byte aligned", fn, !aligned(Y, 4) ? "Y" : "route_w");
    const int S = T * top_k;
    const int64_t Ne = m->N / n_experts;
    // Per-slot outputs straight into Y unless the slots are summed with
    // their routing weights afterwards.
    const bool combine = route_w && !route_on_input;
    MoeScratch ms;
    st = moe_scratch(*m, S, n_experts, combine ? size_t(S) * Ne : 0, 0, fn, ms);
    if (st != QMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = qmm::launch_moe_bucket(expert_ids, S, n_experts, ms.ix, combine ? nullptr : Y,
                                           Ne, Ne, m->status, s);
    if (e == cudaSuccess) {
        qmm::MoeExpertArgs a;
        memset(&a, 0, sizeof(a));
        a.tmap[0] = m->fmt == QMM_Q8_0 ? m->tmap_moe : m->tmap;
        a.y[0] = combine ? ms.ys : Y;
        a.xscale = route_on_input ? route_w : nullptr;
        a.nmat = 1;
        a.Ne = Ne;
        a.K = m->K;
        a.x = X;
        a.ldx = m->K;
        a.top_k = top_k;
        a.x_per_slot = x_per_slot;
        a.ix = ms.ix;
        a.status = m->status;
        e = m->fmt == QMM_Q8_0 ? qmm::launch_moe_q8(a, m->sm_count, s)
                               : qmm::launch_moe_expert(a, m->sm_count, s);
    }
    if (e == cudaSuccess && combine)
        e = qmm::launch_moe_combine(ms.ys, route_w, expert_ids, n_experts, T, top_k, Ne, Y,
                                    m->sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    m->last_stream = s;
    return QMM_OK;
}

qmm_status qmm_swiglu(const float *g, const float *u, float *hh, int64_t n, qmm_stream stream)
{
    g_err.clear();
    const char *fn = "qmm_swiglu";
    if (!g || !u || !hh)
        return fail(QMM_ERR_NULL, "%s: %s is NULL", fn, !g ? "g" : (!u ? "u" : "h"));
    if (n < 0)
        return fail(QMM_ERR_SHAPE, "%s: n = %lld is negative", fn, (long long)n);
    if (!aligned(g, 4) || !aligned(u, 4) || !aligned(hh, 4))
        return fail(QMM_ERR_ALIGN, "%s: g, u and h must be 4-byte aligned", fn);
    if (n == 0)
        return QMM_OK;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = qmm::launch_swiglu(g, u, hh, n, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    return QMM_OK;
}

qmm_status qmm_moe_ffn(qmm_t hg, qmm_t hu, qmm_t hd, int32_t n_experts,
                       const int32_t *expert_ids, int32_t T, int32_t top_k, const float *X,
                       const float *route_w, int32_t route_on_input, float *Y,
                       qmm_stream stream)
{
    g_err.clear();
    const char *fn = "qmm_moe_ffn";
    qmm_status st = check_handle(hg, fn);
    if (st == QMM_OK)
        st = check_handle(hu, fn);
    if (st == QMM_OK)
        st = check_handle(hd, fn);
    if (st != QMM_OK)
        return st;
    Matrix *mg = reinterpret_cast<Matrix *>(hg);
    const Matrix *mu = reinterpret_cast<const Matrix *>(hu);
    const Matrix *md = reinterpret_cast<const Matrix *>(hd);
    st = moe_check(*mg, n_experts, expert_ids, T, top_k, fn);
    if (st == QMM_OK)
        st = moe_check(*mu, n_experts, expert_ids, T, top_k, fn);
    if (st == QMM_OK)
        st = moe_check(*md, n_experts, expert_ids, T, top_k, fn);
    if (st != QMM_OK)
        return st;
    const int64_t d_ff = mg->N / n_experts, d_model = mg->K;
    if (mu->fmt != mg->fmt)
        return fail(QMM_ERR_FORMAT, "%s: gate (format %d) and up (format %d) must share a format "
                    "(they run in one launch)", fn, mg->fmt, mu->fmt);
    if (mu->N != mg->N || mu->K != mg->K || md->K != d_ff || md->N != int64_t(n_experts) * d_model)
        return fail(QMM_ERR_SHAPE,
                    "%s: shapes disagree: gate %lld x %lld, up %lld x %lld, down %lld x %lld; "
                    "with %d experts gate and up must be (E*d_ff) x d_model and down "
                    "(E*d_model) x d_ff",
                    fn, (long long)mg->N, (long long)mg->K, (long long)mu->N, (long long)mu->K,
                    (long long)md->N, (long long)md->K, n_experts);
    if (!X || !Y || !route_w)
        return fail(QMM_ERR_NULL, "%s: %s is NULL", fn, !X ? "X" : (!Y ? "Y" : "route_w"));
    if (route_on_input != 0 && route_on_input != 1)
        return fail(QMM_ERR_SHAPE, "%s: route_on_input = %d; it must be 0 or 1", fn,
                    route_on_input);
    if (!aligned(X, 16))
        return fail(QMM_ERR_ALIGN, "%s: X is not 16-byte aligned", fn);
    if (!aligned(Y, 4) || !aligned(route_w, 4))
        return fail(QMM_ERR_ALIGN, "%s: %s is not 4-byte aligned", fn, !aligned(Y, 4) ? "Y" : "route_w");
    const int S = T * top_k;
    MoeScratch ms;
    st = moe_scratch(*mg, S, n_experts, size_t(S) * d_model, size_t(S) * d_ff, fn, ms);
    if (st != QMM_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = mg->sm_count;
    cudaError_t e = qmm::launch_moe_bucket(expert_ids, S, n_experts, ms.ix, nullptr, 0, 0,
                                           mg->status, s);
    qmm::MoeExpertArgs a;
    memset(&a, 0, sizeof(a));
    a.top_k = top_k;
    a.ix = ms.ix;
    a.status = mg->status;
    // Gate and up in one launch.  With room in shared memory for every CTA's
    // (gate, up) tile pairs, SwiGLU is applied in the same launch; otherwise
    // a separate kernel combines the two products.
    int nw = 0, nslot = 0;
    qmm::moe_expert_shape(d_model, nw, nslot);
    const int64_t tpm = (d_ff + 15) / 16;
    const int maxpairs =
        int((int64_t(qmm::moe_max_groups(S, n_experts)) * tpm + sms - 1) / sms) + 1;
    const bool q8 = mg->fmt == QMM_Q8_0;
    const bool fuse = !getenv("QMM_MOE_NOFUSE") &&
                      (q8 || qmm::moe_expert_smem(d_model, nw, nslot, maxpairs) <= kMaxSmem);
    if (e == cudaSuccess) {
        a.tmap[0] = q8 ? mg->tmap_moe : mg->tmap;
        a.tmap[1] = q8 ? mu->tmap_moe : mu->tmap;
        a.y[0] = fuse ? ms.h : ms.g;
        a.y[1] = fuse ? nullptr : ms.u;
        a.nmat = 2;
        a.Ne = d_ff;
        a.K = d_model;
        a.x = X;
        a.ldx = d_model;
        a.x_per_slot = 0;
        a.xscale = route_on_input ? route_w : nullptr;
        a.fuse_swiglu = fuse ? 1 : 0;
        a.maxpairs = maxpairs;
        e = q8 ? qmm::launch_moe_q8(a, sms, s) : qmm::launch_moe_expert(a, sms, s);
    }
    if (e == cudaSuccess && !fuse)
        e = qmm::launch_swiglu(ms.g, ms.u, ms.h, int64_t(S) * d_ff, sms, s);
    a.fuse_swiglu = 0;
    a.xscale = nullptr;
    if (e == cudaSuccess) {  // down, one input row per slot
        a.tmap[0] = md->fmt == QMM_Q8_0 ? md->tmap_moe : md->tmap;
        a.tmap[1] = nullptr;
        a.y[0] = ms.ys;
        a.y[1] = nullptr;
        a.nmat = 1;
        a.Ne = d_model;
        a.K = d_ff;
        a.x = ms.h;
        a.ldx = d_ff;
        a.x_per_slot = 1;
        e = md->fmt == QMM_Q8_0 ? qmm::launch_moe_q8(a, sms, s) : qmm::launch_moe_expert(a, sms, s);
    }
    if (e == cudaSuccess)
        e = qmm::launch_moe_combine(ms.ys, route_on_input ? nullptr : route_w, expert_ids,
                                    n_experts, T, top_k, d_model, Y, sms, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    mg->last_stream = s;
    return QMM_OK;
}

qmm_status qmm_ffn_decode(qmm_t hg, qmm_t hu, qmm_t hd, const float *x, float *h, float *y,
                          qmm_stream stream)
{
    g_err.clear();
    const char *fn = "qmm_ffn_decode";
    qmm_status st = check_handle(hg, fn);
    if (st == QMM_OK)
        st = check_handle(hu, fn);
    if (st == QMM_OK)
        st = check_handle(hd, fn);
    if (st != QMM_OK)
        return st;
    const Matrix &mg = *reinterpret_cast<const Matrix *>(hg);
    const Matrix &mu = *reinterpret_cast<const Matrix *>(hu);
    const Matrix &md = *reinterpret_cast<const Matrix *>(hd);
    if (mg.fmt != mu.fmt || mg.N != mu.N || mg.K != mu.K || md.K != mg.N)
        return fail(QMM_ERR_SHAPE,
                    "%s: gate %lld x %lld and up %lld x %lld must match (same format too) and down's "
                    "K = %lld must equal their N", fn, (long long)mg.N, (long long)mg.K,
                    (long long)mu.N, (long long)mu.K, (long long)md.K);
    if (!x || !h || !y)
        return fail(QMM_ERR_NULL, "%s: %s is NULL", fn, !x ? "x" : (!h ? "h" : "y"));
    if (!aligned(x, 16) || !aligned(h, 16))
        return fail(QMM_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, !aligned(x, 16) ? "x" : "h");
    if (!aligned(y, 4))
        return fail(QMM_ERR_ALIGN, "%s: y is not 4-byte aligned", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const qmm_t gu[2] = {hg, hu};
    const bool nofuse = getenv("QMM_FFN_NOFUSE") && getenv("QMM_FFN_NOFUSE")[0] == '1';
    // Gate and up on the decode kernel with SwiGLU in its output phase (the
    // pair's tiles interleaved), where it takes the shape; QMM_FFN_PATH=tc
    // keeps the earlier tensor-core kernel's pair mode.
    const char *fpath = getenv("QMM_FFN_PATH");
    st = QMM_ERR_UNSUPPORTED;
    if (!nofuse && !(fpath && strcmp(fpath, "tc") == 0)) {
        float *ys2[2] = {h, nullptr};
        st = do_gemv_m1(gu, 2, x, ys2, s, fn, true);
        if (st != QMM_OK && st != QMM_ERR_UNSUPPORTED)
            return st;
    }
    if (st == QMM_OK) {
        // h written by the fused launch
    } else if (mg.fmt == QMM_Q4_K && tc_fits(mg, 1) && !nofuse) {
        // Gate and up in one tensor-core launch, SwiGLU in its epilogue.
        qmm::TcArgs a;
        memset(&a, 0, sizeof(a));
        a.tmap[0] = mg.tmap;
        a.tmap[1] = mu.tmap;
        a.rows[0] = a.rows[1] = mg.N;
        a.y[0] = h;
        a.nmat = 2;
        a.K = mg.K;
        a.M = 1;
        a.ldx = mg.K;
        a.x = x;
        a.status = mg.status;
        a.fuse_swiglu = 1;
        cudaError_t e = qmm::launch_gemv_tc(a, mg.sm_count, s);
        if (e != cudaSuccess)
            return cuda_fail(e, fn);
        reinterpret_cast<Matrix *>(hg)->last_stream = s;
    } else {
        // Gate into h and up into the up handle's scratch (one grouped launch
        // when both fit a kernel together), then SwiGLU as its own kernel.
        MoeScratch ms;
        st = moe_scratch(*reinterpret_cast<Matrix *>(hu), 1, 1, 0, size_t(mg.N), fn, ms);
        if (st != QMM_OK)
            return st;
        float *ys[2] = {h, ms.u};
        st = do_gemv(gu, 2, x, ys, s, fn);
        if (st != QMM_OK)
            return st;
        cudaError_t e = qmm::launch_swiglu(h, ms.u, h, mg.N, mg.sm_count, s);
        if (e != cudaSuccess)
            return cuda_fail(e, fn);
    }
    // down: y = Wd h
    float *yd[1] = {y};
    return do_gemv(&hd, 1, h, yd, s, fn);
}

// The prefill GEMM for n Q4_K or n Q8_0 matrices sharing X (n <= 4).
static qmm_status gemm_common(const qmm_t *hs, int n, const uint16_t *X_bf16, int64_t M,
                              float *const *Ys, qmm_stream stream, const char *fn)
{
    for (int i = 0; i < n; ++i) {
        qmm_status st = check_handle(hs[i], fn);
        if (st != QMM_OK)
            return st;
        const Matrix *mi = reinterpret_cast<const Matrix *>(hs[i]);
        if ((mi->fmt != QMM_Q4_K && mi->fmt != QMM_Q8_0) || !mi->has_gemm_maps)
            return fail(QMM_ERR_UNSUPPORTED,
                        "%s: the prefill GEMM takes Q4_K, and Q8_0 rows of whole 256-weight "
                        "groups (matrix %d is format %d, K %lld)", fn, i, mi->fmt,
                        (long long)mi->K);
        if (mi->fmt != reinterpret_cast<const Matrix *>(hs[0])->fmt)
            return fail(QMM_ERR_SHAPE, "%s: matrix %d has format %d, matrix 0 format %d", fn, i,
                        mi->fmt, reinterpret_cast<const Matrix *>(hs[0])->fmt);
        if (mi->K != reinterpret_cast<const Matrix *>(hs[0])->K)
            return fail(QMM_ERR_SHAPE, "%s: matrix %d has K = %lld, matrix 0 K = %lld", fn, i,
                        (long long)mi->K, (long long)reinterpret_cast<const Matrix *>(hs[0])->K);
        if (mi->N > (int64_t(1) << 30))
            return fail(QMM_ERR_SHAPE, "%s: N = %lld rows exceed the GEMM's limit of 2^30", fn,
                        (long long)mi->N);
        if (!Ys[i])
            return fail(QMM_ERR_NULL, "%s: output %d is NULL", fn, i);
        if (!aligned(Ys[i], 4))
            return fail(QMM_ERR_ALIGN, "%s: output %d is not 4-byte aligned", fn, i);
    }
    Matrix *m = reinterpret_cast<Matrix *>(hs[0]);
    if (!X_bf16)
        return fail(QMM_ERR_NULL, "%s: X is NULL", fn);
    if (M < 1 || M > (int64_t(1) << 24))
        return fail(QMM_ERR_SHAPE, "%s: M = %lld; 1 <= M <= 16777216 is supported", fn,
                    (long long)M);
    if (!aligned(X_bf16, 16))
        return fail(QMM_ERR_ALIGN, "%s: X is not 16-byte aligned", fn);
    qmm::GemmArgs a;
    memset(&a, 0, sizeof(a));
    a.fmt = m->fmt;
    int64_t Ntot = 0;
    int tiles256 = 0, tiles128 = 0;
    for (int i = 0; i < n; ++i) {
        const Matrix *mi = reinterpret_cast<const Matrix *>(hs[i]);
        a.tmap_hdr[i] = mi->tmap_hdr;
        a.tmap_nib[i] = mi->tmap_nib;
        a.y[i] = Ys[i];
        a.N[i] = mi->N;
        Ntot += mi->N;
        tiles256 += qmm::gemm_q4k_tiles(M, mi->N, 256);
        tiles128 += qmm::gemm_q4k_tiles(M, mi->N, 128);
    }
    a.nmat = n;
    // 256-token tiles reuse each dequantised weight twice as often as 128-token
    // tiles; measured on the Llama shapes at 512 and 2048 tokens they are as
    // fast or faster for every matrix (the K split of the tail wave recovers
    // the parallelism of few tiles).  At most 128 tokens take 128-token tiles
    // (a 256-token tile would be half padding).  QMM_GEMM_TOK forces either.
    a.tok = M <= 128 ? 128 : 256;
    if (const char *e = getenv("QMM_GEMM_TOK"))
        if (atoi(e) == 128 || atoi(e) == 256)
            a.tok = atoi(e);
    const int tiles = a.tok == 128 ? tiles128 : tiles256;
    alignas(64) unsigned char tmx[128];
    if (qmm::encode_tmap_2d(tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X_bf16, uint64_t(m->K),
                            uint64_t(M), uint64_t(m->K) * 2, 64u, uint32_t(a.tok),
                            CU_TENSOR_MAP_SWIZZLE_128B) != 0)
        return fail(QMM_ERR_CUDA, "%s: the TMA tensor map for X could not be encoded", fn);
    const qmm::GemmSplit split = qmm::gemm_q4k_split(tiles, a.tok, m->K, m->sm_count);
    a.ksplit = split.ksplit;
    a.full_tiles = split.full;
    if (a.ksplit > 1) {
        // Split K: the partial products; the scratch of matrix 0 grows on
        // demand (waiting for the device first).
        const size_t need = qmm::gemm_q4k_ws_floats(M, Ntot, a.ksplit) * 4;
        if (need > m->gemm_ws_bytes) {
            cudaError_t e = cudaSuccess;
            if (m->gemm_ws) {
                e = cudaDeviceSynchronize();
                if (e == cudaSuccess)
                    e = cudaFree(m->gemm_ws);
                m->gemm_ws = nullptr;
                m->gemm_ws_bytes = 0;
                if (e != cudaSuccess)
                    return cuda_fail(e, fn);
            }
            void *p = nullptr;
            e = cudaMalloc(&p, need);
            if (e != cudaSuccess)
                return fail(QMM_ERR_NOMEM, "%s: could not allocate %zu bytes of split-K scratch (%s)",
                            fn, need, cudaGetErrorString(e));
            m->gemm_ws = p;
            m->gemm_ws_bytes = need;
        }
        a.ws = static_cast<float *>(m->gemm_ws);
    }
    a.tmap_x = tmx;
    a.M = M;
    a.K = m->K;
    a.status = m->status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = qmm::launch_gemm_q4k(a, m->sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    m->last_stream = s;
    return QMM_OK;
}

qmm_status qmm_gemm(qmm_t h, const uint16_t *X_bf16, int64_t M, float *Y, qmm_stream stream)
{
    g_err.clear();
    return gemm_common(&h, 1, X_bf16, M, &Y, stream, "qmm_gemm");
}

qmm_status qmm_gemm_group(const qmm_t *hs, int32_t n, const uint16_t *X_bf16, int64_t M,
                          float *const *Ys, qmm_stream stream)
{
    g_err.clear();
    if (!hs || !Ys)
        return fail(QMM_ERR_NULL, "qmm_gemm_group: the %s array is NULL", !hs ? "handle" : "output");
    if (n < 1 || n > qmm::kGemmMaxGroup)
        return fail(QMM_ERR_SHAPE, "qmm_gemm_group: n = %d; between 1 and %d matrices are supported",
                    n, qmm::kGemmMaxGroup);
    return gemm_common(hs, n, X_bf16, M, Ys, stream, "qmm_gemm_group");
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

qmm_status qmm_quantize_q8_k(const float *x, int64_t K, void *xq, qmm_stream stream)
{
    g_err.clear();
    const char *fn = "qmm_quantize_q8_k";
    if (!x || !xq)
        return fail(QMM_ERR_NULL, "%s: %s is NULL", fn, !x ? "x" : "xq");
    if (K < 256 || K % 256)
        return fail(QMM_ERR_SHAPE, "%s: K = %lld; a positive multiple of 256 is required", fn,
                    (long long)K);
    if (K / 256 > (int64_t(1) << 30))
        return fail(QMM_ERR_SHAPE, "%s: K = %lld is too large", fn, (long long)K);
    if (!aligned(x, 16) || !aligned(xq, 4))
        return fail(QMM_ERR_ALIGN, "%s: x must be 16-byte and xq 4-byte aligned", fn);
    cudaError_t e = qmm::launch_quantize_q8k(x, K, static_cast<uint8_t *>(xq),
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    return QMM_OK;
}

} // extern "C"

namespace {

// The integer-dot GEMV for n matrices: on Q8_K blocks xq, or (x non-null)
// on f32 activations quantized inside the launch.
qmm_status q8k_group_common(const qmm_t *hs, int32_t n, const void *xq, const float *x,
                            float *const *ys, qmm_stream stream, const char *fn)
{
    if (!hs || !ys)
        return fail(QMM_ERR_NULL, "%s: the %s array is NULL", fn, !hs ? "handle" : "output");
    if (n < 1 || n > qmm::kMaxGroup)
        return fail(QMM_ERR_SHAPE, "%s: n = %d; between 1 and %d matrices are supported", fn,
                    int(n), qmm::kMaxGroup);
    qmm::Q8kArgs a;
    memset(&a, 0, sizeof(a));
    for (int i = 0; i < n; ++i) {
        qmm_status st = check_handle(hs[i], fn);
        if (st != QMM_OK)
            return st;
        const Matrix &mi = *reinterpret_cast<const Matrix *>(hs[i]);
        if (mi.fmt != QMM_Q4_K)
            return fail(QMM_ERR_UNSUPPORTED,
                        "%s: matrix %d has format %d; the integer-dot path takes Q4_K", fn, i,
                        mi.fmt);
        if (mi.K != reinterpret_cast<const Matrix *>(hs[0])->K)
            return fail(QMM_ERR_SHAPE, "%s: matrix %d has K %lld, matrix 0 K %lld", fn, i,
                        (long long)mi.K, (long long)reinterpret_cast<const Matrix *>(hs[0])->K);
        if (!ys[i])
            return fail(QMM_ERR_NULL, "%s: output %d is NULL", fn, i);
        if (!aligned(ys[i], 4))
            return fail(QMM_ERR_ALIGN, "%s: output %d is not 4-byte aligned", fn, i);
        a.w[i] = mi.w;
        a.y[i] = ys[i];
        a.N[i] = mi.N;
    }
    if (x) {
        if (!aligned(x, 16))
            return fail(QMM_ERR_ALIGN, "%s: x is not 16-byte aligned", fn);
    } else {
        if (!xq)
            return fail(QMM_ERR_NULL, "%s: xq is NULL", fn);
        if (!aligned(xq, 4))
            return fail(QMM_ERR_ALIGN, "%s: xq is not 4-byte aligned", fn);
    }
    const Matrix &m0 = *reinterpret_cast<const Matrix *>(hs[0]);
    if (qmm::q8k_smem(m0.K) > size_t(kMaxSmem))
        return fail(QMM_ERR_SHAPE, "%s: K = %lld; its Q8_K activations (%zu bytes) exceed shared "
                                   "memory", fn, (long long)m0.K, qmm::q8k_smem(m0.K));
    a.nmat = n;
    a.K = m0.K;
    a.xq = static_cast<const uint8_t *>(xq);
    a.x = x;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = qmm::launch_gemv_q8k(a, m0.sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, fn);
    reinterpret_cast<Matrix *>(hs[0])->last_stream = s;
    return QMM_OK;
}

} // namespace

extern "C" {

qmm_status qmm_gemv_q8k_group(const qmm_t *hs, int32_t n, const void *xq, float *const *ys,
                              qmm_stream stream)
{
    g_err.clear();
    return q8k_group_common(hs, n, xq, nullptr, ys, stream, "qmm_gemv_q8k_group");
}

qmm_status qmm_gemv_q8k(qmm_t h, const void *xq, float *y, qmm_stream stream)
{
    return qmm_gemv_q8k_group(&h, 1, xq, &y, stream);
}

qmm_status qmm_gemv_q8k_fused_group(const qmm_t *hs, int32_t n, const float *x,
                                    float *const *ys, qmm_stream stream)
{
    g_err.clear();
    if (!x)
        return fail(QMM_ERR_NULL, "qmm_gemv_q8k_fused_group: x is NULL");
    return q8k_group_common(hs, n, nullptr, x, ys, stream, "qmm_gemv_q8k_fused_group");
}

qmm_status qmm_gemv_q8k_fused(qmm_t h, const float *x, float *y, qmm_stream stream)
{
    g_err.clear();
    if (!x)
        return fail(QMM_ERR_NULL, "qmm_gemv_q8k_fused: x is NULL");
    return q8k_group_common(&h, 1, nullptr, x, &y, stream, "qmm_gemv_q8k_fused");
}

} // extern "C"
