"""GPU parity of the further block formats (Q5_K, Q6_K, IQ4_NL) against the
oracle, through the C ABI: block decode bit-exact (fp32 = RN_fp32 of the
exact weight, bf16 = RN_even of that fp32 value), the decode GEMV and the
batched GEMV within 1e-4 of sum|w x|, the dense FFN through its grouped
route, and the refusals of the calls that take Q4_K only."""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests._util import TOL_FP32, assert_close_to_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("quantized_gguf_dequant_gb300")

FORMATS = [q.Q5_K, q.Q6_K, q.IQ4_NL]
NT = max(1, oracle.max_threads())


def _matrix(fmt, N, K, seed):
    w = synth.matrix(fmt, N, K, seed)
    return w, q.Matrix(fmt, N, K, to_dev(w))


@pytest.mark.parametrize("fmt", FORMATS)
def test_dequant_bit_exact(fmt):
    N, K = 7, 768
    w, m = _matrix(fmt, N, K, seed=100 + fmt)
    ref = oracle.dequant_rows(fmt, w, N, K).astype(np.float32)  # RN_fp32 of the exact values
    got = m.dequantize().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    part = m.dequantize(row0=3, nrows=2).cpu().numpy()
    assert np.array_equal(part.view(np.uint32), ref[3:5].view(np.uint32))
    bf = m.dequantize_bf16().cpu().numpy().view(np.uint16)
    ref_bf = np.array([[oracle.bf16_from_float(v) for v in row] for row in ref], dtype=np.uint16)
    assert np.array_equal(bf, ref_bf)
    m.close()


@pytest.mark.parametrize("path", ["default", "staged", "fast", "plain"])
@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N,K", [(1, 256), (9, 512), (300, 2048), (4096, 4096), (33, 768),
                                 (77, 14336), (5, 8192), (1000, 6144)])
def test_gemv(monkeypatch, path, fmt, N, K):
    """The one-row GEMV on every route: the staged fp32 kernel (where its
    32-lane teams fit, K-sliced for long rows; the SIMT kernel elsewhere),
    the SIMT kernel (1, 2, 3, 16, 24, 32 and 56 units per row), the plain
    one, and the default choice among them."""
    if path != "default":
        monkeypatch.setenv("QMM_FMT_PATH", path)
    w, m = _matrix(fmt, N, K, seed=N + K + fmt)
    x = synth.activations(1, K, seed=K + 1)[0]
    y = m.gemv(to_dev(x)).cpu().numpy()
    yr, c = oracle.gemv(fmt, w, N, K, x, nthreads=NT)
    assert_close_to_oracle(y, yr, c, TOL_FP32, f"fmt={fmt} N={N} K={K}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M", [1, 3, 16])
def test_gemv_batched(fmt, M):
    N, K = 77, 1024
    w, m = _matrix(fmt, N, K, seed=M + fmt)
    X = synth.activations(M, K, seed=M + 5)
    Y = m.gemv_batched(to_dev(X)).cpu().numpy()
    Yr, C = oracle.gemv(fmt, w, N, K, X, nthreads=NT)
    assert_close_to_oracle(Y, Yr, C, TOL_FP32, f"fmt={fmt} M={M}")
    # a repeated call gives the same bits; so does one row at a time on the
    # same (SIMT) kernel
    Y2 = m.gemv_batched(to_dev(X)).cpu().numpy()
    assert np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))
    os.environ["QMM_FMT_PATH"] = "fast"
    try:
        y0 = m.gemv(to_dev(X[0])).cpu().numpy()
    finally:
        del os.environ["QMM_FMT_PATH"]
    assert np.array_equal(Y[0].view(np.uint32), y0.view(np.uint32))
    m.close()


def test_gemv_group_mixed_with_q4k_down_in_ffn():
    """A dense FFN whose gate/up are Q5_K and whose down is Q6_K (a mix the
    K-quant files use), through qmm_ffn_decode's grouped route."""
    d_model, d_ff = 512, 768
    wg, hg = _matrix(q.Q5_K, d_ff, d_model, seed=1)
    wu, hu = _matrix(q.Q5_K, d_ff, d_model, seed=2)
    wd, hd = _matrix(q.Q6_K, d_model, d_ff, seed=3)
    x = synth.activations(1, d_model, seed=4)[0]
    h = torch.full((d_ff,), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((d_model,), float("nan"), dtype=torch.float32, device="cuda")
    q.ffn_decode(hg.h, hu.h, hd.h, to_dev(x), h, y)
    torch.cuda.synchronize()
    g, cg = oracle.gemv(q.Q5_K, wg, d_ff, d_model, x[None], nthreads=NT)
    u, cu = oracle.gemv(q.Q5_K, wu, d_ff, d_model, x[None], nthreads=NT)
    h_ref = oracle.swiglu(g[0], u[0])
    sg = oracle.swiglu(g[0], np.ones_like(g[0]))
    a = np.abs(h_ref) + 1.1 * np.abs(u[0]) * cg[0] + np.abs(sg) * cu[0]
    assert_close_to_oracle(h.cpu().numpy(), h_ref, a * 1.0001, TOL_FP32, "h")
    y_ref, _ = oracle.gemv(q.Q6_K, wd, d_model, d_ff, h_ref.astype(np.float32)[None], nthreads=NT)
    _, cd = oracle.gemv(q.Q6_K, wd, d_model, d_ff, a.astype(np.float32)[None], nthreads=NT)
    assert_close_to_oracle(y.cpu().numpy(), y_ref[0], cd[0] * 1.0001, TOL_FP32, "y")
    for m in (hg, hu, hd):
        m.close()


def test_q4k_only_calls_refuse():
    w, m = _matrix(q.Q6_K, 64, 256, seed=9)
    X = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
    Y = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        m.gemm(X, Y)
    assert ei.value.status in (q.ERR_UNSUPPORTED, q.ERR_FORMAT)
    ids = torch.zeros((2, 1), dtype=torch.int32, device="cuda")
    Xm = torch.zeros((2, 256), dtype=torch.float32, device="cuda")
    Ym = torch.zeros((2, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.moe_gemv(m.h, 2, ids, 2, 1, Xm, False, None, Ym)
    assert ei.value.status in (q.ERR_UNSUPPORTED, q.ERR_FORMAT)
    m.close()


@pytest.mark.parametrize("fmt", [q.Q8_0, q.IQ4_NL])
@pytest.mark.parametrize("N,K", [(37, 32), (300, 4128), (77, 96), (5, 14368)])
def test_block32_formats_with_k_not_a_multiple_of_256(fmt, N, K):
    """32-weight-block formats take any K that fills whole blocks: rows are
    then only 2-byte aligned, and the per-group kernels read them bytewise.
    GEMV, batched GEMV, a group of two, decode and bf16 decode."""
    w, m = _matrix(fmt, N, K, seed=N + K + fmt)
    X = synth.activations(3, K, seed=K + 2)
    yr, c = oracle.gemv(fmt, w, N, K, X, nthreads=NT)
    y = m.gemv(to_dev(X[0])).cpu().numpy()
    assert_close_to_oracle(y, yr[0], c[0], TOL_FP32, f"gemv fmt={fmt} K={K}")
    Y = torch.full((3, N), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_batched(m.h, to_dev(X), 3, K, Y, N)
    torch.cuda.synchronize()
    assert_close_to_oracle(Y.cpu().numpy(), yr, c, TOL_FP32, f"batched fmt={fmt} K={K}")
    w2, m2 = _matrix(fmt, 11, K, seed=N + K + fmt + 1)
    y1 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    y2 = torch.full((11,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_group([m.h, m2.h], to_dev(X[1]), [y1, y2])
    torch.cuda.synchronize()
    assert_close_to_oracle(y1.cpu().numpy(), yr[1], c[1], TOL_FP32, "group 0")
    yr2, c2 = oracle.gemv(fmt, w2, 11, K, X[1], nthreads=NT)
    assert_close_to_oracle(y2.cpu().numpy(), yr2, c2, TOL_FP32, "group 1")
    ref = oracle.dequant_rows(fmt, w, N, K).astype(np.float32)
    got = m.dequantize().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert m.status() == 0
    m.close()
    m2.close()


def test_q8_0_noalloc_with_k_not_a_multiple_of_256():
    N, K = 300, 4128
    w = synth.matrix(q.Q8_0, N, K, seed=17)
    x = synth.activations(1, K, seed=18)[0]
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_noalloc(q.Q8_0, N, K, to_dev(w), to_dev(x), y)
    torch.cuda.synchronize()
    yr, c = oracle.gemv(q.Q8_0, w, N, K, x, nthreads=NT)
    assert_close_to_oracle(y.cpu().numpy(), yr, c, TOL_FP32, "noalloc Q8_0 K=4128")


def test_create_refusals():
    w = torch.zeros(1000, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.Matrix(q.Q6_K, 1, 100, w)  # K not a multiple of 256
    assert ei.value.status == q.ERR_SHAPE
    with pytest.raises(q.QmmError) as ei:
        q.Matrix(q.Q8_0, 1, 100, w)  # K not a multiple of 32
    assert ei.value.status == q.ERR_SHAPE
    with pytest.raises(q.QmmError) as ei:
        q.Matrix(15, 1, 256, w)  # Q8_K: not a weight format here
    assert ei.value.status == q.ERR_FORMAT


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_group_fast(fmt):
    """q/k/v-like group of three matrices sharing x in one fast launch, and
    the result bitwise equal on a second call."""
    K = 2048
    Ns = [512, 128, 128]
    ws, ms = zip(*[_matrix(fmt, N, K, seed=50 + i + fmt) for i, N in enumerate(Ns)])
    x = synth.activations(1, K, seed=60)[0]
    outs = []
    for _ in range(2):
        ys = [torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
        q.gemv_group([m.h for m in ms], to_dev(x), ys)
        torch.cuda.synchronize()
        outs.append([y.cpu().numpy() for y in ys])
    for i, (N, w) in enumerate(zip(Ns, ws)):
        yr, c = oracle.gemv(fmt, w, N, K, x, nthreads=NT)
        assert_close_to_oracle(outs[0][i], yr, c, TOL_FP32, f"group {i}")
        assert np.array_equal(outs[0][i].view(np.uint32), outs[1][i].view(np.uint32))
    for m in ms:
        m.close()
