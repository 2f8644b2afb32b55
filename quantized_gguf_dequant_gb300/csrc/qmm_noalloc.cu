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
#include <mutex>

#include "qmm_internal.h"

namespace {

// Layout of the static scratch: [status word, padded to 256 B][tickets]
// [split-K partial sums].  1 MiB in total; every GPU that loads the library
// keeps it until the process exits.
constexpr size_t kScratchBytes = size_t(1) << 20;
constexpr size_t kStatusBytes = 256;
constexpr size_t kTickets = 4096;
constexpr size_t kPartialFloats = (kScratchBytes - kStatusBytes - kTickets * 4) / 4;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// The device address of g_scratch on the current device, looked up once per
// device (the host-side name is only a stand-in for it).
cudaError_t scratch_address(int dev, void **out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess)
            return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
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
    if (dev < 0 || dev >= kMaxDevices)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: device %d is beyond the %d "
                                               "devices this entry point tracks", dev, kMaxDevices);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: %s", cudaGetErrorString(e));
    const qmm::GemvPlan p = qmm::plan_gemv(fmt, N, K, sms, 0);
    const size_t need = qmm::gemv_workspace_floats(p, N);
    if (need > kPartialFloats || size_t(p.row_slices) > kTickets)
        return qmm::noalloc_fail(
            QMM_ERR_SHAPE,
            "qmm_gemv_noalloc: this shape needs %zu floats of split-K scratch and %d tickets; the "
            "static scratch holds %zu floats and %zu tickets (use qmm_create/qmm_gemv)",
            need, p.row_slices, kPartialFloats, kTickets);
    void *base = nullptr;
    e = scratch_address(dev, &base);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA,
                                 "qmm_gemv_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
                                 cudaGetErrorString(e));
    unsigned char *b = static_cast<unsigned char *>(base);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The tickets must start at zero.  A completed call leaves them zero, but
    // a call that timed out may not, so clear them (and the status word) on
    // the stream first -- a memset, not an allocation.
    e = cudaMemsetAsync(b, 0, kStatusBytes + size_t(p.row_slices) * 4, s);
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
    a.tickets = reinterpret_cast<unsigned *>(b + kStatusBytes);
    a.ws = reinterpret_cast<float *>(b + kStatusBytes + kTickets * 4);
    e = qmm::launch_gemv(p, a, s);
    if (e != cudaSuccess)
        return qmm::noalloc_fail(QMM_ERR_CUDA, "qmm_gemv_noalloc: launch failed: %s",
                                 cudaGetErrorString(e));
    return QMM_OK;
}

} // extern "C"
