"""Seeded random shapes through every compute entry point, against the oracle.

Each case draws the weight format, N, K (any multiple of 256), batch sizes,
expert counts and top-k from a fixed seed, so odd row counts (not multiples
of 16 or 256), odd super-block counts and odd batch sizes all occur; each
result must meet the path's bound (1e-4 of sum|w x| for the fp32 paths, 1e-3
for the bf16 prefill against the oracle's bf16 product).  QMM_FUZZ_SEED
shifts every seed and QMM_FUZZ_CASES sets the number of cases, for longer
runs than the default 12 cases of seed 0."""
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

NT = max(1, oracle.max_threads())
CASES = int(os.environ.get("QMM_FUZZ_CASES", "12"))
SHIFT = 100000 * int(os.environ.get("QMM_FUZZ_SEED", "0"))


def _rng(case, salt):
    return np.random.default_rng(SHIFT + 1000 * salt + case)


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_gemv_and_batched(case):
    r = _rng(case, 1)
    fmt = [q.Q4_K, q.Q8_0, q.Q4_K, q.Q5_K, q.Q6_K, q.IQ4_NL][int(r.integers(0, 6))]
    N = int(r.integers(1, 700))
    K = 256 * int(r.integers(1, 24))
    M = int(r.integers(1, 17))
    w = synth.matrix(fmt, N, K, SHIFT + 50 + case)
    m = q.Matrix(fmt, N, K, to_dev(w))
    X = synth.activations(M, K, SHIFT + 60 + case)
    Y = m.gemv_batched(to_dev(X)).cpu().numpy()
    y1 = m.gemv(to_dev(X[0])).cpu().numpy()
    Yr, C = oracle.gemv(fmt, w, N, K, X, nthreads=NT)
    assert_close_to_oracle(Y, Yr, C, TOL_FP32, f"batched fmt={fmt} N={N} K={K} M={M}")
    assert_close_to_oracle(y1, Yr[0], C[0], TOL_FP32, f"gemv fmt={fmt} N={N} K={K}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_gemm(case):
    r = _rng(case, 2)
    fmt = q.Q8_0 if r.integers(0, 3) == 0 else q.Q4_K
    N = int(r.integers(1, 900))
    K = 256 * int(r.integers(1, 12))
    M = int(r.integers(1, 600))
    w = synth.matrix(fmt, N, K, SHIFT + 70 + case)
    m = q.Matrix(fmt, N, K, to_dev(w))
    Xb = synth.activations_bf16(M, K, SHIFT + 80 + case)
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    m.gemm(to_dev(Xb.view(np.int16)), Y)
    torch.cuda.synchronize()
    Yr, C = oracle.gemm_bf16(w, N, K, Xb, nthreads=NT, fmt=fmt)
    assert_close_to_oracle(Y.cpu().numpy(), Yr, C, 1e-3, f"gemm fmt={fmt} N={N} K={K} M={M}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_moe(case):
    r = _rng(case, 3)
    fmt = q.Q8_0 if r.integers(0, 3) == 0 else q.Q4_K
    E = int(r.integers(1, 24))
    Ne = int(r.integers(1, 200))
    K = 256 * int(r.integers(1, 6))
    T = int(r.integers(1, 40))
    top_k = int(r.integers(1, min(E, 8) + 1))
    xps = bool(case % 2)
    routed = case % 3 != 0
    w = synth.matrix(fmt, E * Ne, K, SHIFT + 90 + case)
    m = q.Matrix(fmt, E * Ne, K, to_dev(w))
    ids, rw = synth.router(T, E, top_k, SHIFT + 91 + case)
    X = synth.activations(T * top_k if xps else T, K, SHIFT + 92 + case)
    rows = T if routed else T * top_k
    Y = torch.full((rows, Ne), float("nan"), dtype=torch.float32, device="cuda")
    q.moe_gemv(m.h, E, to_dev(ids), T, top_k, to_dev(X), xps, to_dev(rw) if routed else None, Y)
    torch.cuda.synchronize()
    Yr, C = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, xps, rw if routed else None, nthreads=NT)
    assert_close_to_oracle(Y.cpu().numpy(), Yr, C, TOL_FP32,
                           f"moe fmt={fmt} E={E} Ne={Ne} K={K} T={T} k={top_k} xps={xps} routed={routed}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_ffn_decode(case):
    """qmm_ffn_decode on random widths and formats (the decode kernel's fused
    gate/up pairs, or the grouped route where they do not fit), against the
    oracle composition with the GEMV bound carried through SwiGLU."""
    r = _rng(case, 4)
    fmt = [q.Q4_K, q.Q8_0, q.Q5_K, q.Q6_K, q.IQ4_NL][int(r.integers(0, 5))]
    d_model = 256 * int(r.integers(1, 20))
    d_ff = 256 * int(r.integers(1, 30))
    wg = synth.matrix(fmt, d_ff, d_model, SHIFT + 110 + case)
    wu = synth.matrix(fmt, d_ff, d_model, SHIFT + 111 + case)
    wd = synth.matrix(fmt, d_model, d_ff, SHIFT + 112 + case)
    x = synth.activations(1, d_model, SHIFT + 113 + case)[0]
    hs = [q.Matrix(fmt, d_ff, d_model, to_dev(wg)), q.Matrix(fmt, d_ff, d_model, to_dev(wu)),
          q.Matrix(fmt, d_model, d_ff, to_dev(wd))]
    h = torch.full((d_ff,), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((d_model,), float("nan"), dtype=torch.float32, device="cuda")
    q.ffn_decode(hs[0].h, hs[1].h, hs[2].h, to_dev(x), h, y)
    torch.cuda.synchronize()
    g, cg = oracle.gemv(fmt, wg, d_ff, d_model, x[None], nthreads=NT)
    u, cu = oracle.gemv(fmt, wu, d_ff, d_model, x[None], nthreads=NT)
    h_ref = oracle.swiglu(g[0], u[0])
    sg = oracle.swiglu(g[0], np.ones_like(g[0]))
    a = np.abs(h_ref) + 1.1 * np.abs(u[0]) * cg[0] + np.abs(sg) * cu[0]
    what = f"ffn fmt={fmt} d_model={d_model} d_ff={d_ff}"
    assert_close_to_oracle(h.cpu().numpy(), h_ref, a * 1.0001, TOL_FP32, what + " h")
    y_ref, _ = oracle.gemv(fmt, wd, d_model, d_ff, h_ref.astype(np.float32)[None], nthreads=NT)
    _, cd = oracle.gemv(fmt, wd, d_model, d_ff, a.astype(np.float32)[None], nthreads=NT)
    assert_close_to_oracle(y.cpu().numpy(), y_ref[0], cd[0] * 1.0001, TOL_FP32, what + " y")
    for m in hs:
        assert m.status() == 0
        m.close()


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_gemv_group(case):
    """qmm_gemv_group: one to four matrices of random, ragged row counts that
    share x, in one format, each against the oracle."""
    r = _rng(case, 5)
    fmt = [q.Q4_K, q.Q8_0, q.Q5_K, q.Q6_K, q.IQ4_NL][int(r.integers(0, 5))]
    K = 256 * int(r.integers(1, 40))
    Ns = [int(r.integers(1, 1500)) for _ in range(int(r.integers(1, 5)))]
    ws = [synth.matrix(fmt, N, K, SHIFT + 120 + 10 * case + i) for i, N in enumerate(Ns)]
    ms = [q.Matrix(fmt, N, K, to_dev(w)) for N, w in zip(Ns, ws)]
    x = synth.activations(1, K, SHIFT + 121 + case)[0]
    ys = [torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
    q.gemv_group([m.h for m in ms], to_dev(x), ys)
    torch.cuda.synchronize()
    for i, (N, w, y) in enumerate(zip(Ns, ws, ys)):
        yr, c = oracle.gemv(fmt, w, N, K, x, nthreads=NT)
        assert_close_to_oracle(y.cpu().numpy(), yr, c, TOL_FP32, f"group {i} fmt={fmt} N={Ns} K={K}")
    for m in ms:
        assert m.status() == 0
        m.close()


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_gemv_q8k(case):
    """The opt-in integer-dot GEMV on random shapes: the quantizer's bytes
    equal the oracle's, the GEMV is within 1e-5 of sum|w xhat| of the
    oracle's integer-dot GEMV, and the variant that quantizes inside the
    launch gives the same bits."""
    r = _rng(case, 6)
    N = int(r.integers(1, 3000))
    K = 256 * int(r.integers(1, 60))
    w = synth.q4k_matrix(N, K, SHIFT + 130 + case)
    x = synth.activations(1, K, SHIFT + 131 + case)[0]
    xq_ref = oracle.quantize_q8_k(x)
    xq = torch.full((K // 256 * q.Q8_K_BLOCK,), 0xAB, dtype=torch.uint8, device="cuda")
    q.quantize_q8_k(to_dev(x), K, xq)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), np.asarray(xq_ref, dtype=np.uint8))
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_q8k(m.h, xq, y)
    yf = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_q8k_fused(m.h, to_dev(x), yf)
    torch.cuda.synchronize()
    y_ref, c = oracle.gemv_q8k(q.Q4_K, w, N, K, xq_ref, nthreads=NT)
    got = y.cpu().numpy()
    assert_close_to_oracle(got, y_ref, c, 1e-5, f"q8k N={N} K={K}")
    assert np.array_equal(got.view(np.int32), yf.cpu().numpy().view(np.int32))
    assert m.status() == 0
    m.close()
