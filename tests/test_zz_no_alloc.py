"""The decode GEMV entry point for callers that cannot allocate device memory.

qmm_gemv_noalloc takes the matrix description instead of a handle and keeps
its split-K scratch in a fixed array inside the library, so a caller that may
not call cudaMalloc (a fixed memory pool, a driver-managed allocator, a
plug-in that must not grow the process's device footprint) can still run the
product.  Checked here through the C ABI against the allocating entry point
(qmm_create + qmm_gemv) on two calls in a row: the shared scratch keeps the
previous call's contents, and the second call must still be right.  This file
sorts last so that a run stopping at the first failure has run every other
test before it; it also passes alone in a fresh process (the first call on a
device does the one-time scratch lookup).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests._util import TOL_FP32, assert_close_to_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("quantized_gguf_dequant_gb300")


@pytest.mark.parametrize("fmt", [q.Q4_K, q.Q8_0])
@pytest.mark.parametrize("N,K", [(37, 2048), (3000, 4096), (5, 14336)])
def test_noalloc_matches_allocating_gemv_twice(fmt, N, K):
    w = synth.matrix(fmt, N, K, seed=500 + N)
    wd = to_dev(w)
    m = q.Matrix(fmt, N, K, wd)
    for call in range(2):
        x = synth.activations(1, K, seed=600 + N + call)[0]
        xd = to_dev(x)
        y_alloc = m.gemv(xd).cpu().numpy()
        y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        q.gemv_noalloc(fmt, N, K, wd, xd, y)
        got = y.cpu().numpy()
        _, c = oracle.gemv(fmt, w, N, K, x)
        assert_close_to_oracle(got, y_alloc, c, TOL_FP32, f"noalloc vs allocating, call {call}")
    m.close()


def test_noalloc_refuses_oversized_scratch():
    # N x K that would need more split-K scratch than the fixed array holds:
    # refused on the host, before anything runs (the pointers are never read).
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    y = torch.zeros(16, dtype=torch.float32, device="cuda")
    rc = q.lib().qmm_gemv_noalloc(q.Q4_K, 4096, 1 << 20, ctypes.c_void_p(buf.data_ptr()),
                                  ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == q.ERR_SHAPE
    assert "static scratch holds" in q.last_error()
