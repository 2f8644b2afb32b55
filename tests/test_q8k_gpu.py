"""GPU parity of the integer-dot variant (Q8_K activations) through the C ABI.

"Frink Inference: the Rust alternative to llama.cpp", section "Where
llama.cpp is still ahead": llama.cpp quantizes activations to Q8_K before a
K-quant dot product.  Checked here:

* qmm_quantize_q8_k: the Q8_K bytes, bit-exact against the oracle's
  quantizer (the codes are decided in binary32 on both sides).
* qmm_gemv_q8k / _group: against the oracle's integer-dot GEMV (the exact
  weights times the exact dequantized activations, fp64), within
  1e-5 * sum |w xhat| -- the integer partial sums are exact, only the fp32
  scaling per super-block and the fp32 sum round.
* The drift against the f32 path stays inside the stated bound:
  |y_q8k - y_f32| <= sum_b (sum over block b of |w|) * |d_b| / 2.
"""
from __future__ import annotations

import ctypes
import struct

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests._util import assert_close_to_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("quantized_gguf_dequant_gb300")

TOL_Q8K = 1e-5
NTHREADS = max(1, oracle.max_threads())


def _quantize_dev(x: np.ndarray) -> torch.Tensor:
    K = x.size
    xq = torch.full((K // 256 * q.Q8_K_BLOCK,), 0xAB, dtype=torch.uint8, device="cuda")
    q.quantize_q8_k(to_dev(x.astype(np.float32)), K, xq)
    torch.cuda.synchronize()
    return xq


def _special_blocks() -> np.ndarray:
    """Blocks that exercise the quantizer's decisions: all zero, ties to
    even, equal magnitudes of both signs (first wins), a negative and a
    positive max, tiny and huge scales, signed zeros."""
    blocks = []
    z = np.zeros(256, np.float32)
    blocks.append(z.copy())
    b = z.copy()
    b[0], b[1], b[2], b[3], b[4] = -63.5, 0.25, 0.75, 1.25, -1.25  # iscale = 2
    blocks.append(b)
    b = z.copy()
    b[3], b[10] = -4.0, 4.0
    blocks.append(b)
    b = z.copy()
    b[200], b[17] = 4.0, -4.0
    blocks.append(b)
    b = z.copy()
    b[5], b[6], b[7], b[20], b[255] = -1.0, 0.5, -0.25, 0.75, 1.0 / 127.0
    blocks.append(b)
    rng = np.random.default_rng(7)
    blocks.append((rng.standard_normal(256) * 1e-30).astype(np.float32))
    blocks.append((rng.standard_normal(256) * 1e30).astype(np.float32))
    b = z.copy()
    b[::2] = -0.0
    b[100] = 3.0
    blocks.append(b)
    blocks.append(np.full(256, -2.5, np.float32))
    return np.concatenate(blocks)


@pytest.mark.parametrize("K", [256, 2048, 4096, 14336])
def test_quantize_bit_exact(K):
    x = synth.activations(1, K, seed=K)[0]
    got = _quantize_dev(x).cpu().numpy()
    assert np.array_equal(got, oracle.quantize_q8_k(x))


def test_quantize_special_blocks_bit_exact():
    x = _special_blocks()
    got = _quantize_dev(x).cpu().numpy()
    ref = oracle.quantize_q8_k(x)
    for b in range(x.size // 256):
        assert np.array_equal(got[292 * b:292 * (b + 1)], ref[292 * b:292 * (b + 1)]), b


@pytest.mark.parametrize("N,K", [
    (1, 256), (37, 2048), (300, 4096), (77, 14336), (4096, 4096),
    (5, 8192),      # 32 super-blocks: one row per warp, one per lane
    (3, 768),       # 3 super-blocks: lanes stride, most idle
    (10, 1280),     # 5 super-blocks
    (33, 512),      # 2 super-blocks: 16 rows per warp, ragged tail
])
def test_gemv_q8k_matches_oracle(N, K):
    w = synth.q4k_matrix(N, K, seed=N + K)
    x = synth.activations(1, K, seed=N * 3 + 1)[0]
    xq = oracle.quantize_q8_k(x)
    y_ref, c = oracle.gemv_q8k(q.Q4_K, w, N, K, xq, nthreads=NTHREADS)
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_q8k(m.h, _quantize_dev(x), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    assert_close_to_oracle(got, y_ref, c, TOL_Q8K, f"q8k {N}x{K}")
    # bitwise repeatable
    y2 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_q8k(m.h, _quantize_dev(x), y2)
    torch.cuda.synchronize()
    assert np.array_equal(got.view(np.int32), y2.cpu().numpy().view(np.int32))
    # quantized inside the GEMV launch: the same bits
    y3 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_q8k_fused(m.h, to_dev(x), y3)
    torch.cuda.synchronize()
    assert np.array_equal(got.view(np.int32), y3.cpu().numpy().view(np.int32))
    m.close()


def test_gemv_q8k_drift_within_stated_bound():
    """Against the f32 oracle: the GPU result of the integer path stays
    within the stated drift bound plus its own fp32 tolerance."""
    N, K = 512, 4096
    w = synth.q4k_matrix(N, K, seed=91)
    x = synth.activations(1, K, seed=92)[0]
    xq = oracle.quantize_q8_k(x)
    y32, _ = oracle.gemv(q.Q4_K, w, N, K, x, nthreads=NTHREADS)
    _, c8 = oracle.gemv_q8k(q.Q4_K, w, N, K, xq, nthreads=NTHREADS)
    W = np.abs(oracle.dequant_rows(q.Q4_K, w, N, K)).reshape(N, K // 256, 256).sum(axis=2)
    dq = np.array([abs(struct.unpack("<f", xq[292 * b:292 * b + 4].tobytes())[0])
                   for b in range(K // 256)])
    bound = W @ (dq * (0.5 + 2.0 ** -20)) + TOL_Q8K * c8
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    q.gemv_q8k(m.h, _quantize_dev(x), y)
    torch.cuda.synchronize()
    drift = np.abs(y.cpu().numpy().astype(np.float64) - y32)
    assert np.all(drift <= bound)
    m.close()


def test_gemv_q8k_group():
    """q/k/v of Llama-3.1-8B sharing one quantized input, in one launch."""
    K = 4096
    shapes = [4096, 1024, 1024]
    ws = [synth.q4k_matrix(N, K, seed=120 + i) for i, N in enumerate(shapes)]
    x = synth.activations(1, K, seed=123)[0]
    xq = oracle.quantize_q8_k(x)
    ms = [q.Matrix(q.Q4_K, N, K, to_dev(w)) for N, w in zip(shapes, ws)]
    ys = [torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for N in shapes]
    q.gemv_q8k_group([m.h for m in ms], _quantize_dev(x), ys)
    yf = [torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for N in shapes]
    q.gemv_q8k_fused_group([m.h for m in ms], to_dev(x), yf)
    torch.cuda.synchronize()
    for N, w, y, y2 in zip(shapes, ws, ys, yf):
        y_ref, c = oracle.gemv_q8k(q.Q4_K, w, N, K, xq, nthreads=NTHREADS)
        assert_close_to_oracle(y.cpu().numpy(), y_ref, c, TOL_Q8K, f"group N={N}")
        assert np.array_equal(y.cpu().numpy().view(np.int32), y2.cpu().numpy().view(np.int32))
    for m in ms:
        m.close()


@pytest.mark.parametrize("K", [256, 4096, 14336])
def test_gemv_q8k_fused_special_blocks(K):
    """The in-launch quantization on blocks with a zero block, ties of the
    largest magnitude and extreme scales: the same bits as the separate
    quantization."""
    N = 40
    w = synth.q4k_matrix(N, K, seed=K + 7)
    x = synth.activations(1, K, seed=K + 8)[0]
    x[:256] = 0.0                      # a zero block
    if K > 256:
        x[256:512] = np.float32(1e-30) * x[256:512]
        amax = np.abs(x[256:512]).max()
        x[300], x[301] = -amax, amax  # ties in magnitude: the first one sets the sign
    x[-256:] *= np.float32(1e30)
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    y1 = torch.empty(N, dtype=torch.float32, device="cuda")
    y2 = torch.empty(N, dtype=torch.float32, device="cuda")
    q.gemv_q8k(m.h, _quantize_dev(x), y1)
    q.gemv_q8k_fused(m.h, to_dev(x), y2)
    torch.cuda.synchronize()
    assert np.array_equal(y1.cpu().numpy().view(np.int32), y2.cpu().numpy().view(np.int32))
    m.close()


def test_q8k_in_cuda_graph():
    """quantize + GEMV captured in a CUDA graph replay to the eager bits."""
    N, K = 1000, 4096
    w = synth.q4k_matrix(N, K, seed=130)
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    x = to_dev(synth.activations(1, K, seed=131)[0])
    xq = torch.empty(K // 256 * q.Q8_K_BLOCK, dtype=torch.uint8, device="cuda")
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q.quantize_q8_k(x, K, xq, s)
        q.gemv_q8k(m.h, xq, y, s)
    s.synchronize()
    eager = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q.quantize_q8_k(x, K, xq, s)
        q.gemv_q8k(m.h, xq, y, s)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), eager.view(torch.int32))
    m.close()


def test_q8k_refusals():
    K = 512
    w8 = synth.matrix(q.Q8_0, 4, K, seed=1)
    m8 = q.Matrix(q.Q8_0, 4, K, to_dev(w8))
    x = to_dev(synth.activations(1, K, seed=2)[0])
    xq = torch.zeros(K // 256 * q.Q8_K_BLOCK + 8, dtype=torch.uint8, device="cuda")
    y = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.gemv_q8k(m8.h, xq, y)
    assert ei.value.status == q.ERR_UNSUPPORTED
    with pytest.raises(q.QmmError) as ei:
        q.quantize_q8_k(x, 300, xq)
    assert ei.value.status == q.ERR_SHAPE
    rc = q.lib().qmm_quantize_q8_k(ctypes.c_void_p(x.data_ptr()), K,
                                   ctypes.c_void_p(xq.data_ptr() + 2), None)
    assert rc == q.ERR_ALIGN
    w4 = synth.q4k_matrix(4, K, seed=3)
    w4b = synth.q4k_matrix(4, 2 * K, seed=4)
    m4, m4b = q.Matrix(q.Q4_K, 4, K, to_dev(w4)), q.Matrix(q.Q4_K, 4, 2 * K, to_dev(w4b))
    with pytest.raises(q.QmmError) as ei:
        q.gemv_q8k_group([m4.h, m4b.h], xq, [y, y])
    assert ei.value.status == q.ERR_SHAPE
    for m in (m8, m4, m4b):
        m.close()
