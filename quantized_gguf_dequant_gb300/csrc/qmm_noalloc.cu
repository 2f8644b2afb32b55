// qmm_noalloc.cu -- the decode GEMV for callers that cannot allocate device
// memory: no handle, no cudaMalloc.  Its scratch (split-K partial sums,
// per-row-range tickets and the device status word) lives in one fixed,
// file-scope device array that the library image carries.
//
// Who needs this: code that runs where cudaMalloc is unavailable or unwanted
// -- inside a host callback or a driver-managed allocator, in a process whose
// memory pool is fixed up front, or in a plug-in that must not change the
// host program's device-memory footprint after start-up.
#include <cstring>

#include "qmm_internal.h"

namespace {

using qmm::kNoallocPartialFloats;
using qmm::kNoallocScratchBytes;
using qmm::kNoallocStatusBytes;
using qmm::kNoallocTickets;

static __device__ __align__(256) unsigned char g_scratch[kNoallocScratchBytes];

// The device address of g_scratch in the current context, looked up on every
// call: a context torn down and made again (cudaDeviceReset) may place the
// image elsewhere, so no address is kept between calls.
cudaError_t scratch_address(void **out)
{
    return cudaGetSymbolAddress(out, g_scratch);
}

} // namespace

extern "C" {

qmm_status qmm_gemv_noalloc(qmm_format fmt, int64_t N, int64_t K, const void *w_dev,
                            const float *x, float *y, qmm_stream stream)
{
    qmm_status st = qmm::noalloc_check(fmt, N, K, w_dev, x, y);
    if (st != QMM_OK)
        return st;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: cudaGetDevice failed: %s",
                                 cudaGetErrorString(e));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fmt == QMM_Q8_0 && K % 256 != 0) {
        // Rows of whole 32-weight blocks that are not whole 256-weight groups:
        // the per-group kernel, one warp per row, no scratch at all.
        qmm::Matrix m;
        m.fmt = fmt;
        m.N = N;
        m.K = K;
        m.row_bytes = qmm::row_bytes_of(fmt, K);
        m.w = static_cast<const uint8_t *>(w_dev);
        e = qmm::launch_gemv_fmt(m, x, 1, K, y, N, s);
        if (e != cudaSuccess)
            return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: launch failed: %s",
                                     cudaGetErrorString(e));
        return QMM_OK;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: %s", cudaGetErrorString(e));
    const qmm::GemvPlan p = qmm::plan_gemv(fmt, N, K, sms, 0);
    const size_t need = qmm::gemv_workspace_floats(p, N);
    if (!qmm::noalloc_fits(p, N))
        return qmm::noalloc_fail(
            QMM_ERR_SHAPE,
            "qmm_gemv_noalloc: this shape needs %zu floats of split-K scratch and %d tickets; the "
            "static scratch holds %zu floats and %zu tickets (use qmm_create/qmm_gemv)",
            need, p.row_slices, kNoallocPartialFloats, kNoallocTickets);
    void *base = nullptr;
    e = scratch_address(&base);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA,
                                 "qmm_gemv_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
                                 cudaGetErrorString(e));
    unsigned char *b = static_cast<unsigned char *>(base);
    // The tickets must start at zero.  A completed call leaves them zero, but
    // a call that timed out may not, so clear them (and the status word) on
    // the stream first -- a memset, not an allocation.
    e = cudaMemsetAsync(b, 0, kNoallocStatusBytes + size_t(p.row_slices) * 4, s);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: clearing the scratch failed: %s",
                                 cudaGetErrorString(e));
    qmm::GemvArgs a;
    memset(&a, 0, sizeof(a));
    a.fmt = fmt;
    a.nmat = 1;
    a.w[0] = static_cast<const uint8_t *>(w_dev);
    a.y[0] = y;
    for (int i = 0; i < qmm::kMaxGroup; ++i)
        a.row_end[i] = N;
    a.N = N;
    a.K = K;
    a.row_bytes = qmm::row_bytes_of(fmt, K);
    a.x = x;
    a.status = reinterpret_cast<unsigned *>(b);
    a.tickets = reinterpret_cast<unsigned *>(b + kNoallocStatusBytes);
    a.ws = reinterpret_cast<float *>(b + kNoallocStatusBytes + kNoallocTickets * 4);
    e = qmm::launch_gemv(p, a, s);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: launch failed: %s",
                                 cudaGetErrorString(e));
    return QMM_OK;
}

} // extern "C"
