"""Fused-dequantisation GGUF quantized matmul for one GB300 (sm_103a).

A thin ctypes binding over libqmm.so, the C ABI declared in include/qmm.h.
It only marshals arguments: torch tensors supply device memory and the
current CUDA stream, and every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if libqmm.so is missing or cannot be
loaded, every call raises.

Names follow the C ABI (``qmm_gemv`` -> ``gemv`` and so on).  ``Matrix`` owns
a handle for a quantized weight tensor kept on the device.
"""
from __future__ import annotations

import ctypes
import os

Q8_0 = 8
Q4_K = 12
Q5_K = 13
Q6_K = 14
IQ4_NL = 20

OK = 0
ERR_NULL, ERR_FORMAT, ERR_SHAPE, ERR_ALIGN, ERR_CUDA = -1, -2, -3, -4, -5
ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_NOMEM, ERR_EXPERT = -6, -7, -8, -9

_HERE = os.path.dirname(os.path.abspath(__file__))
# QMM_LIBRARY may name another build of the library (e.g. an instrumented one).
LIB_PATH = os.environ.get("QMM_LIBRARY") or os.path.join(_HERE, "libqmm.so")
_lib = None

# Every entry point of include/qmm.h.
ENTRY_POINTS = (
    "qmm_create", "qmm_destroy", "qmm_gemv", "qmm_gemv_group", "qmm_gemv_batched",
    "qmm_moe_gemv", "qmm_swiglu", "qmm_moe_ffn", "qmm_gemm", "qmm_dequantize",
    "qmm_dequantize_bf16", "qmm_get_status", "qmm_last_error", "qmm_version",
    "qmm_gemv_noalloc", "qmm_gemm_group", "qmm_launch_count", "qmm_ffn_decode",
    "qmm_quantize_q8_k", "qmm_gemv_q8k", "qmm_gemv_q8k_group", "qmm_gemv_q8k_fused",
    "qmm_gemv_q8k_fused_group",
)


class QmmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status
        self.message = message


def lib() -> ctypes.CDLL:
    """The loaded libqmm.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m quantized_gguf_dequant_gb300.build` (there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        sig = {
            "qmm_create": [i32, i64, i64, vp, ctypes.POINTER(vp)],
            "qmm_destroy": [vp],
            "qmm_gemv": [vp, vp, vp, vp],
            "qmm_gemv_group": [ctypes.POINTER(vp), i32, vp, ctypes.POINTER(vp), vp],
            "qmm_gemv_batched": [vp, vp, i64, i64, vp, i64, vp],
            "qmm_moe_gemv": [vp, i32, vp, i32, i32, vp, i32, vp, i32, vp, vp],
            "qmm_swiglu": [vp, vp, vp, i64, vp],
            "qmm_moe_ffn": [vp, vp, vp, i32, vp, i32, i32, vp, vp, i32, vp, vp],
            "qmm_gemm": [vp, vp, i64, vp, vp],
            "qmm_dequantize": [vp, i64, i64, vp, vp],
            "qmm_dequantize_bf16": [vp, i64, i64, vp, vp],
            "qmm_get_status": [vp],
            "qmm_last_error": [],
            "qmm_version": [],
            "qmm_gemv_noalloc": [i32, i64, i64, vp, vp, vp, vp],
            "qmm_gemm_group": [ctypes.POINTER(vp), i32, vp, i64, ctypes.POINTER(vp), vp],
            "qmm_ffn_decode": [vp, vp, vp, vp, vp, vp, vp],
            "qmm_quantize_q8_k": [vp, i64, vp, vp],
            "qmm_gemv_q8k": [vp, vp, vp, vp],
            "qmm_gemv_q8k_group": [ctypes.POINTER(vp), i32, vp, ctypes.POINTER(vp), vp],
            "qmm_gemv_q8k_fused": [vp, vp, vp, vp],
            "qmm_gemv_q8k_fused_group": [ctypes.POINTER(vp), i32, vp, ctypes.POINTER(vp), vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = i32
        L.qmm_last_error.restype = ctypes.c_char_p
        L.qmm_launch_count.argtypes = []
        L.qmm_launch_count.restype = ctypes.c_int64
        _lib = L
    return _lib


def last_error() -> str:
    return lib().qmm_last_error().decode()


def version() -> int:
    return int(lib().qmm_version())


def launch_count() -> int:
    """Kernel launches the library has issued in this process so far."""
    return int(lib().qmm_launch_count())


def _check(rc: int):
    if rc != OK:
        raise QmmError(rc, last_error())


def _ptr(t) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("tensor must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None) -> ctypes.c_void_p:
    import torch
    if stream is None:
        # the current stream's handle without building a Stream object
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return ctypes.c_void_p(raw(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# --------------------------------------------------------------------- raw ABI

def create(fmt: int, N: int, K: int, w) -> int:
    h = ctypes.c_void_p()
    _check(lib().qmm_create(fmt, N, K, _ptr(w), ctypes.byref(h)))
    return h.value


def destroy(h: int):
    _check(lib().qmm_destroy(ctypes.c_void_p(h)))


def gemv(h: int, x, y, stream=None):
    _check(lib().qmm_gemv(ctypes.c_void_p(h), _ptr(x), _ptr(y), _stream(stream)))


def gemv_group(hs, x, ys, stream=None):
    n = len(hs)
    harr = (ctypes.c_void_p * n)(*[ctypes.c_void_p(h) for h in hs])
    yarr = (ctypes.c_void_p * n)(*[_ptr(y) for y in ys])
    _check(lib().qmm_gemv_group(harr, n, _ptr(x), yarr, _stream(stream)))


def gemv_batched(h: int, X, M: int, ldx: int, Y, ldy: int, stream=None):
    _check(lib().qmm_gemv_batched(ctypes.c_void_p(h), _ptr(X), M, ldx, _ptr(Y), ldy,
                                  _stream(stream)))


def moe_gemv(h: int, n_experts: int, ids, T: int, top_k: int, X, x_per_slot: int,
             route_w, Y, stream=None, route_on_input: bool = False):
    _check(lib().qmm_moe_gemv(ctypes.c_void_p(h), n_experts, _ptr(ids), T, top_k, _ptr(X),
                              int(x_per_slot), _ptr(route_w), int(route_on_input), _ptr(Y),
                              _stream(stream)))


def ffn_decode(hg: int, hu: int, hd: int, x, h, y, stream=None):
    """qmm_ffn_decode: h = silu(Wg x) * (Wu x), y = Wd h (one token)."""
    _check(lib().qmm_ffn_decode(ctypes.c_void_p(hg), ctypes.c_void_p(hu), ctypes.c_void_p(hd),
                                _ptr(x), _ptr(h), _ptr(y), _stream(stream)))


def swiglu(g, u, hout, n: int, stream=None):
    _check(lib().qmm_swiglu(_ptr(g), _ptr(u), _ptr(hout), n, _stream(stream)))


def moe_ffn(hg: int, hu: int, hd: int, n_experts: int, ids, T: int, top_k: int, X, route_w, Y,
            stream=None, route_on_input: bool = False):
    _check(lib().qmm_moe_ffn(ctypes.c_void_p(hg), ctypes.c_void_p(hu), ctypes.c_void_p(hd),
                             n_experts, _ptr(ids), T, top_k, _ptr(X), _ptr(route_w),
                             int(route_on_input), _ptr(Y), _stream(stream)))


Q8_K_BLOCK = 292  # bytes per 256 activations in the Q8_K encoding


def quantize_q8_k(x, K: int, xq, stream=None):
    """qmm_quantize_q8_k: K fp32 activations -> K/256 Q8_K blocks in xq."""
    _check(lib().qmm_quantize_q8_k(_ptr(x), K, _ptr(xq), _stream(stream)))


def gemv_q8k(h: int, xq, y, stream=None):
    """qmm_gemv_q8k: the integer-dot GEMV of a Q4_K matrix with Q8_K activations."""
    _check(lib().qmm_gemv_q8k(ctypes.c_void_p(h), _ptr(xq), _ptr(y), _stream(stream)))


def gemv_q8k_group(hs, xq, ys, stream=None):
    n = len(hs)
    harr = (ctypes.c_void_p * n)(*[ctypes.c_void_p(h) for h in hs])
    yarr = (ctypes.c_void_p * n)(*[_ptr(y) for y in ys])
    _check(lib().qmm_gemv_q8k_group(harr, n, _ptr(xq), yarr, _stream(stream)))


def gemv_q8k_fused(h: int, x, y, stream=None):
    """qmm_gemv_q8k_fused: the integer-dot GEMV on f32 activations, quantized
    to Q8_K inside the launch."""
    _check(lib().qmm_gemv_q8k_fused(ctypes.c_void_p(h), _ptr(x), _ptr(y), _stream(stream)))


def gemv_q8k_fused_group(hs, x, ys, stream=None):
    n = len(hs)
    harr = (ctypes.c_void_p * n)(*[ctypes.c_void_p(h) for h in hs])
    yarr = (ctypes.c_void_p * n)(*[_ptr(y) for y in ys])
    _check(lib().qmm_gemv_q8k_fused_group(harr, n, _ptr(x), yarr, _stream(stream)))


def gemm(h: int, X_bf16, M: int, Y, stream=None):
    _check(lib().qmm_gemm(ctypes.c_void_p(h), _ptr(X_bf16), M, _ptr(Y), _stream(stream)))


def gemm_group(hs, X_bf16, M: int, Ys, stream=None):
    n = len(hs)
    harr = (ctypes.c_void_p * n)(*[ctypes.c_void_p(h) for h in hs])
    yarr = (ctypes.c_void_p * n)(*[_ptr(y) for y in Ys])
    _check(lib().qmm_gemm_group(harr, n, _ptr(X_bf16), M, yarr, _stream(stream)))


def dequantize(h: int, row0: int, nrows: int, out, stream=None):
    _check(lib().qmm_dequantize(ctypes.c_void_p(h), row0, nrows, _ptr(out), _stream(stream)))


def dequantize_bf16(h: int, row0: int, nrows: int, out, stream=None):
    _check(lib().qmm_dequantize_bf16(ctypes.c_void_p(h), row0, nrows, _ptr(out),
                                     _stream(stream)))


def gemv_noalloc(fmt: int, N: int, K: int, w, x, y, stream=None):
    """qmm_gemv_noalloc: the decode GEMV without a handle or any device
    allocation (scratch lives in a fixed array inside the library)."""
    _check(lib().qmm_gemv_noalloc(fmt, N, K, _ptr(w), _ptr(x), _ptr(y), _stream(stream)))


def get_status(h: int) -> int:
    """The handle's device status (0 = OK); clears it."""
    return int(lib().qmm_get_status(ctypes.c_void_p(h)))


# --------------------------------------------------------------------- wrapper

class Matrix:
    """A quantized N x K matrix on the device (a torch uint8 tensor of its
    GGUF bytes) with its library handle."""

    def __init__(self, fmt: int, N: int, K: int, w_dev):
        import torch
        if w_dev.dtype != torch.uint8:
            raise ValueError("weights must be a uint8 tensor of GGUF block bytes")
        self.fmt, self.N, self.K = fmt, N, K
        self.w = w_dev  # keep the bytes alive as long as the handle
        self.h = create(fmt, N, K, w_dev)

    def close(self):
        if getattr(self, "h", None):
            destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def gemv(self, x, y=None, stream=None):
        import torch
        if y is None:
            y = torch.empty(self.N, dtype=torch.float32, device=x.device)
        gemv(self.h, x, y, stream)
        return y

    def gemv_batched(self, X, Y=None, stream=None):
        import torch
        M = X.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.float32, device=X.device)
        gemv_batched(self.h, X, M, X.stride(0), Y, Y.stride(0), stream)
        return Y

    def gemm(self, X_bf16, Y=None, stream=None):
        import torch
        M = X_bf16.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.float32, device=X_bf16.device)
        gemm(self.h, X_bf16, M, Y, stream)
        return Y

    def dequantize(self, row0=0, nrows=None, out=None, stream=None):
        import torch
        nrows = self.N - row0 if nrows is None else nrows
        if out is None:
            out = torch.empty((nrows, self.K), dtype=torch.float32, device=self.w.device)
        dequantize(self.h, row0, nrows, out, stream)
        return out

    def dequantize_bf16(self, row0=0, nrows=None, out=None, stream=None):
        import torch
        nrows = self.N - row0 if nrows is None else nrows
        if out is None:
            out = torch.empty((nrows, self.K), dtype=torch.int16, device=self.w.device)
        dequantize_bf16(self.h, row0, nrows, out, stream)
        return out

    def status(self) -> int:
        return get_status(self.h)
