"""CPU oracle for the fused-dequant quantized matmul -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never does, and it shares no code with it.

The arithmetic lives in ``qmm_oracle.c`` (plain C, fp64); this module loads
the shared object with ctypes and adds the composite mixture-of-experts
steps, written out in numpy fp64 from the same definitions:

* "Building a Rust Inference Engine That Matches Llama.cpp", sections
  "What Ferrox actually is" / "Where the wins came from": dequantisation is
  fused into the dot product, so the result is the plain decode-then-dot.
* "Frink Inference: the Rust alternative to llama.cpp", section "Where
  llama.cpp is still ahead": activations stay in f32 (no Q8_K).
* Expert routing and the expert FFN (gate, up, SwiGLU, down, routing-weighted
  sum over a token's experts): the OLMoE-style mixture-of-experts layer the
  pages run ("Utility: why this is more than a benchmark exercise").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

Q8_0 = 8
Q4_K = 12
Q5_K = 13
Q6_K = 14
IQ4_NL = 20

# (bytes, weights) of one block of each format
BLOCK = {Q8_0: (34, 32), Q4_K: (144, 256), Q5_K: (176, 256), Q6_K: (210, 256),
         IQ4_NL: (18, 32)}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile qmm_oracle.c into liboracle.so (gcc, OpenMP, ISO C11)."""
    if force or not os.path.exists(_LIB) or (
            os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.or_half_to_double.argtypes = [ctypes.c_uint16]
        L.or_half_to_double.restype = ctypes.c_double
        L.or_q4k_scale_min.argtypes = [vp, i32, vp, vp]
        L.or_dequant_block_q4k.argtypes = [vp, vp]
        L.or_dequant_block_q8_0.argtypes = [vp, vp]
        L.or_dequant_block_q5k.argtypes = [vp, vp]
        L.or_dequant_block_q6k.argtypes = [vp, vp]
        L.or_dequant_block_iq4nl.argtypes = [vp, vp]
        L.or_row_bytes.argtypes = [i32, i64]
        L.or_row_bytes.restype = i64
        L.or_dequant_rows.argtypes = [i32, vp, i64, i64, i64, i64, vp]
        L.or_gemv.argtypes = [i32, vp, i64, i64, vp, i64, i64, vp, i64, vp, vp, i32]
        L.or_gemm_bf16.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, vp, vp, i32]
        L.or_gemm_bf16_fmt.argtypes = [i32, vp, i64, i64, vp, i64, i64, vp, i64, vp, vp, i32]
        L.or_bf16_from_float.argtypes = [ctypes.c_float]
        L.or_bf16_from_float.restype = ctypes.c_uint16
        L.or_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_double.restype = ctypes.c_double
        L.or_swiglu.argtypes = [vp, vp, i64, vp]
        L.or_quantize_q8_k.argtypes = [vp, i64, vp]
        L.or_dequant_q8_k.argtypes = [vp, i64, vp]
        L.or_gemv_q8k.argtypes = [i32, vp, i64, i64, vp, vp, vp, i32]
        L.or_max_threads.restype = i32
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def max_threads() -> int:
    return int(lib().or_max_threads())


# ---------------------------------------------------------------- scalars

def half_to_float64(bits: int) -> float:
    """IEEE binary16 bit pattern -> exact value."""
    return float(lib().or_half_to_double(int(bits) & 0xFFFF))


def q4k_scale_min(sc12: bytes, j: int) -> tuple[int, int]:
    """(scale, min) 6-bit integers of sub-block j of a Q4_K super-block."""
    b = np.frombuffer(bytes(sc12), dtype=np.uint8).copy()
    assert b.size == 12
    sc = ctypes.c_int()
    m = ctypes.c_int()
    _check(lib().or_q4k_scale_min(_p(b), int(j), ctypes.byref(sc), ctypes.byref(m)),
           "q4k_scale_min")
    return sc.value, m.value


def bf16_from_float(f: float) -> int:
    """float -> bfloat16 bit pattern, round to nearest even."""
    return int(lib().or_bf16_from_float(float(np.float32(f))))


def bf16_to_float64(bits: int) -> float:
    return float(lib().or_bf16_to_double(int(bits) & 0xFFFF))


# ---------------------------------------------------------------- decode

def row_bytes(fmt: int, K: int) -> int:
    rb = int(lib().or_row_bytes(fmt, K))
    if rb < 0:
        raise ValueError(f"K={K} does not fill whole blocks of format {fmt}")
    return rb


def dequant_block(fmt: int, block: bytes) -> np.ndarray:
    """The exact values of one block of any supported format."""
    b = np.frombuffer(bytes(block), dtype=np.uint8).copy()
    nbytes, nw = BLOCK[fmt]
    assert b.size == nbytes
    out = np.empty(nw, np.float64)
    fn = {Q4_K: lib().or_dequant_block_q4k, Q8_0: lib().or_dequant_block_q8_0,
          Q5_K: lib().or_dequant_block_q5k, Q6_K: lib().or_dequant_block_q6k,
          IQ4_NL: lib().or_dequant_block_iq4nl}[fmt]
    _check(fn(_p(b), _p(out)), f"dequant_block({fmt})")
    return out


def dequant_rows(fmt: int, w: np.ndarray, N: int, K: int,
                 row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Exact (fp64) weights of rows row0..row0+nrows-1, shape [nrows, K]."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    if nrows is None:
        nrows = N - row0
    assert w.size >= N * row_bytes(fmt, K)
    out = np.empty((nrows, K), np.float64)
    _check(lib().or_dequant_rows(fmt, _p(w), N, K, row0, nrows, _p(out)),
           "dequant_rows")
    return out


# ---------------------------------------------------------------- products

def gemv(fmt: int, w: np.ndarray, N: int, K: int, X: np.ndarray,
         rows=None, nthreads: int = 1):
    """Y[m, i] = sum_k w[rows[i], k] * X[m, k] in fp64; also C = sum |w x|.

    X is fp32 [M, K] (or [K]).  Returns (Y, C), each [M, nrows] (or [nrows]).
    """
    w = np.ascontiguousarray(w, dtype=np.uint8)
    squeeze = X.ndim == 1
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float32)
    M = X.shape[0]
    assert X.shape[1] == K
    assert w.size >= N * row_bytes(fmt, K)
    if rows is None:
        rows_a = None
        nrows = N
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_a.size
    Y = np.empty((M, nrows), np.float64)
    C = np.empty((M, nrows), np.float64)
    _check(lib().or_gemv(fmt, _p(w), N, K, _p(X), M, K,
                         None if rows_a is None else _p(rows_a), nrows,
                         _p(Y), _p(C), int(nthreads)), "gemv")
    if squeeze:
        return Y[0], C[0]
    return Y, C


def gemm_bf16(w: np.ndarray, N: int, K: int, Xbf16: np.ndarray,
              rows=None, nthreads: int = 1, fmt: int = Q4_K):
    """Prefill product with bf16 weights bf16(RN_fp32(w)) and bf16 X.

    Xbf16 holds bfloat16 bit patterns (uint16) [M, K].  Returns (Y, C), each
    [M, nrows]; C is taken with the exact weights.  w is in format fmt.
    """
    w = np.ascontiguousarray(w, dtype=np.uint8)
    X = np.ascontiguousarray(np.atleast_2d(Xbf16), dtype=np.uint16)
    M = X.shape[0]
    assert X.shape[1] == K
    if rows is None:
        rows_a = None
        nrows = N
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_a.size
    Y = np.empty((M, nrows), np.float64)
    C = np.empty((M, nrows), np.float64)
    _check(lib().or_gemm_bf16_fmt(fmt, _p(w), N, K, _p(X), M, K,
                                  None if rows_a is None else _p(rows_a), nrows,
                                  _p(Y), _p(C), int(nthreads)), "gemm_bf16")
    return Y, C


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u with silu(z) = z / (1 + exp(-z)), fp64."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    assert g.shape == u.shape
    h = np.empty_like(g)
    _check(lib().or_swiglu(_p(g), _p(u), g.size, _p(h)), "swiglu")
    return h


# ---------------------------------------------------------------- experts

def moe_gemv(fmt: int, w: np.ndarray, n_experts: int, N_e: int, K: int,
             ids: np.ndarray, X: np.ndarray, x_per_slot: bool,
             route_w: np.ndarray | None = None, nthreads: int = 1,
             route_on_input: bool = False):
    """Grouped expert GEMV driven by router expert ids.

    w holds n_experts matrices of N_e x K stacked back to back (row r of
    expert e is global row e*N_e + r).  ids is [T, top_k].  The input of slot
    (t, s) is X[t] when x_per_slot is False, else X[t*top_k + s].
    Without route_w: returns (Y, C) with Y[t*top_k + s] = W_e x   ([T*top_k, N_e]).
    With route_w [T, top_k]: Y[t] = sum_s r[t,s] * W_{ids[t,s]} x_(t,s),
    C[t] = sum_s |r[t,s]| * sum_k |w x|  ([T, N_e]).
    With route_w and route_on_input (the Llama 4 form: the routing weight
    multiplies the expert's input, "Frink Inference: the Rust alternative to
    llama.cpp", "Architecture coverage: 100 models with evidence"): per slot,
    no sum, Y[t*top_k + s] = W_e (r[t,s] x_(t,s)) with the scaled input
    formed in fp64, C = sum_k |w| |r x|  ([T*top_k, N_e]).
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, top_k = ids.shape
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float32)
    assert X.shape[0] == (T * top_k if x_per_slot else T) and X.shape[1] == K
    if ids.min() < 0 or ids.max() >= n_experts:
        raise ValueError("expert id out of range")
    if route_on_input:
        if route_w is None:
            raise ValueError("route_on_input needs route_w")
        r = np.asarray(route_w, dtype=np.float64).reshape(-1)
        Y = np.zeros((T * top_k, N_e), np.float64)
        C = np.zeros((T * top_k, N_e), np.float64)
        for e in np.unique(ids):
            slots = np.nonzero(ids.reshape(-1) == e)[0]
            xin = (X[slots] if x_per_slot else X[slots // top_k]).astype(np.float64)
            xin = r[slots][:, None] * xin
            W = dequant_rows(fmt, w, n_experts * N_e, K, row0=e * N_e, nrows=N_e)
            Y[slots] = xin @ W.T
            C[slots] = np.abs(xin) @ np.abs(W).T
        return Y, C
    slot_y = np.zeros((T * top_k, N_e), np.float64)
    slot_c = np.zeros((T * top_k, N_e), np.float64)
    rows_of = np.arange(N_e, dtype=np.int64)
    for e in np.unique(ids):
        slots = np.nonzero(ids.reshape(-1) == e)[0]
        xin = X[slots] if x_per_slot else X[slots // top_k]
        Y, C = gemv(fmt, w, n_experts * N_e, K, xin, rows=e * N_e + rows_of,
                    nthreads=nthreads)
        slot_y[slots] = Y
        slot_c[slots] = C
    if route_w is None:
        return slot_y, slot_c
    r = np.asarray(route_w, dtype=np.float64).reshape(T, top_k)
    Y = np.zeros((T, N_e), np.float64)
    C = np.zeros((T, N_e), np.float64)
    for s in range(top_k):
        Y += r[:, s:s + 1] * slot_y.reshape(T, top_k, N_e)[:, s]
        C += np.abs(r[:, s:s + 1]) * slot_c.reshape(T, top_k, N_e)[:, s]
    return Y, C


def moe_ffn(fmt: int, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray,
            n_experts: int, d_model: int, d_ff: int, ids: np.ndarray,
            X: np.ndarray, route_w: np.ndarray, nthreads: int = 1,
            route_on_input: bool = False):
    """The whole expert FFN in fp64: for each token t and slot s with
    e = ids[t,s]:  g = Wg_e x_t, u = Wu_e x_t, h = silu(g) u,
    y_t += r[t,s] * Wd_e h.  Gate/up are d_ff x d_model per expert and down is
    d_model x d_ff.  Returns y [T, d_model] (fp64).

    route_on_input (Llama 4, "Frink Inference: the Rust alternative to
    llama.cpp", "Architecture coverage: 100 models with evidence": the expert
    weight applied to the input of the expert): g = Wg_e (r x_t),
    u = Wu_e (r x_t), h = silu(g) u, y_t += Wd_e h -- r scales the input and
    is not applied again.  SwiGLU is not homogeneous, so the two forms
    differ unless r = 1."""
    ids = np.asarray(ids, dtype=np.int64)
    T, top_k = ids.shape
    if route_on_input:
        g, _ = moe_gemv(fmt, w_gate, n_experts, d_ff, d_model, ids, X, False, route_w,
                        nthreads=nthreads, route_on_input=True)
        u, _ = moe_gemv(fmt, w_up, n_experts, d_ff, d_model, ids, X, False, route_w,
                        nthreads=nthreads, route_on_input=True)
        r = np.ones((T, top_k), np.float64)
    else:
        g, _ = moe_gemv(fmt, w_gate, n_experts, d_ff, d_model, ids, X, False,
                        nthreads=nthreads)
        u, _ = moe_gemv(fmt, w_up, n_experts, d_ff, d_model, ids, X, False,
                        nthreads=nthreads)
        r = np.asarray(route_w, dtype=np.float64).reshape(T, top_k)
    h = swiglu(g, u)
    y = np.zeros((T, d_model), np.float64)
    for e in np.unique(ids):
        slots = np.nonzero(ids.reshape(-1) == e)[0]
        Wd = dequant_rows(fmt, w_down, n_experts * d_model, d_ff,
                          row0=e * d_model, nrows=d_model)
        o = h[slots] @ Wd.T
        for j, sl in enumerate(slots):
            y[sl // top_k] += r[sl // top_k, sl % top_k] * o[j]
    return y


# ---------------------------------------------------------------- Q8_K activations

Q8_K_BLOCK = 292  # bytes per 256 activations: d (f32), q[256] (int8), bsums[16] (int16)


def quantize_q8_k(x: np.ndarray) -> np.ndarray:
    """GGUF Q8_K blocks of the fp32 vector x (len % 256 == 0), as uint8."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(x.size // 256 * Q8_K_BLOCK, np.uint8)
    _check(lib().or_quantize_q8_k(_p(x), x.size, _p(out)), "quantize_q8_k")
    return out


def dequant_q8_k(xq: np.ndarray, K: int) -> np.ndarray:
    """The fp64 activations the Q8_K blocks stand for (d * q)."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    assert xq.size >= K // 256 * Q8_K_BLOCK
    out = np.empty(K, np.float64)
    _check(lib().or_dequant_q8_k(_p(xq), K, _p(out)), "dequant_q8_k")
    return out


def gemv_q8k(fmt: int, w: np.ndarray, N: int, K: int, xq: np.ndarray, nthreads: int = 1):
    """(Y, C): the integer-dot GEMV against Q8_K activations, as the exact
    weights times the exact dequantized activations in fp64."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    Y = np.empty(N, np.float64)
    C = np.empty(N, np.float64)
    _check(lib().or_gemv_q8k(fmt, _p(w), N, K, _p(xq), _p(Y), _p(C), nthreads), "gemv_q8k")
    return Y, C
