"""The decode GEMV entry point for callers that cannot allocate device memory.

qmm_gemv_noalloc takes the matrix description instead of a handle and keeps
its split-K scratch in a fixed array inside the library, so a caller that may
not call cudaMalloc (a fixed memory pool, a driver-managed allocator, a
plug-in that must not grow the process's device footprint) can still run the
product.  Checked here through the C ABI against the oracle on two calls in a
row: the shared scratch keeps the previous call's contents, and the second
call must still be right.  This file sorts last so that a run stopping at the
first failure has run every other test before it; it also passes alone in a
fresh process.
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
def test_noalloc_matches_oracle_twice(fmt, N, K):
    # (37, 2048) and (5, 14336) split K eight ways (the host planner test
    # asserts it), so the partial sums go through the static scratch; two
    # calls in a row, so the second finds the first one's leftovers there.
    w = synth.matrix(fmt, N, K, seed=500 + N)
    wd = to_dev(w)
    m = q.Matrix(fmt, N, K, wd)
    for call in range(2):
        x = synth.activations(1, K, seed=600 + N + call)[0]
        xd = to_dev(x)
        y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        q.gemv_noalloc(fmt, N, K, wd, xd, y)
        got = y.cpu().numpy()
        y_ref, c = oracle.gemv(fmt, w, N, K, x)
        assert_close_to_oracle(got, y_ref, c, TOL_FP32, f"noalloc vs oracle, call {call}")
        y_alloc = m.gemv(xd).cpu().numpy()
        assert_close_to_oracle(y_alloc, y_ref, c, TOL_FP32, f"allocating vs oracle, call {call}")
    m.close()


def test_noalloc_refuses_oversized_scratch():
    # 16384 x 2^20 Q4_K splits K 64 ways: 2^20 floats of partial sums, four
    # times what the fixed array holds -- refused on the host, before
    # anything runs.  The buffers are nonetheless valid for the shape (9.7 GB
    # of weights), so a refusal that stopped working could not touch memory
    # outside them.
    N, K = 16384, 1 << 20
    buf = torch.empty(N * synth.row_bytes(synth.Q4_K, K), dtype=torch.uint8, device="cuda")
    x = torch.zeros(K, dtype=torch.float32, device="cuda")
    y = torch.zeros(N, dtype=torch.float32, device="cuda")
    rc = q.lib().qmm_gemv_noalloc(q.Q4_K, N, K, ctypes.c_void_p(buf.data_ptr()),
                                  ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    del buf
    assert rc == q.ERR_SHAPE
    assert "static scratch holds" in q.last_error()
