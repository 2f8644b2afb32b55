"""GPU parity of the tensor-core prefill GEMM (qmm_gemm) against the CPU
oracle, through the C ABI.

The GEMM multiplies bf16 X by the weights rounded to bf16 (bf16(RN_fp32(w)))
with fp32 accumulation.  The contract bound is |y - y_ref| <= 1e-2 * sum|w x|
(exact weights); since the oracle's y_ref uses the same bf16 weights, the
tests also hold the kernel to 1e-3 of that sum, which only accumulation order
can use up.  An identity X makes Y the transposed bf16 weight matrix, which
must match the oracle's decode bit for bit."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests._util import TOL_BF16, assert_close_to_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("quantized_gguf_dequant_gb300")

NTHREADS = max(1, oracle.max_threads())
TIGHT = 1e-3


def _bf16_bits_of(ref32: np.ndarray) -> np.ndarray:
    """bf16 (nearest even) bit patterns of fp32 values, via torch's CPU cast."""
    t = torch.from_numpy(np.ascontiguousarray(ref32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _run(m, Xb, M):
    Y = torch.full((M, m.N), float("nan"), dtype=torch.float32, device="cuda")
    m.gemm(to_dev(Xb.view(np.int16)), Y)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


def _check(M, N, K, seed, rows=None, fmt=None):
    fmt = q.Q4_K if fmt is None else fmt
    w = synth.matrix(fmt, N, K, seed)
    Xb = synth.activations_bf16(M, K, seed + 1)
    m = q.Matrix(fmt, N, K, to_dev(w))
    y = _run(m, Xb, M)
    y_ref, c = oracle.gemm_bf16(w, N, K, Xb, rows=rows, nthreads=NTHREADS, fmt=fmt)
    got = y if rows is None else y[:, rows]
    assert_close_to_oracle(got, y_ref, c, TOL_BF16, f"gemm M={M} N={N} K={K}")
    assert_close_to_oracle(got, y_ref, c, TIGHT, f"gemm (tight) M={M} N={N} K={K}")
    assert m.status() == 0
    m.close()
    return y


@pytest.mark.parametrize("fmt", [12, 8])  # Q4_K, Q8_0
def test_gemm_identity_is_bf16_weights(fmt):
    """X = I (K x K): Y[m][n] = bf16(w[n][m]) exactly (one nonzero product per
    output), for every position of every super-block, chunk and nibble (Q8_0:
    every block and code of every 80-byte window offset)."""
    N, K = 300, 512
    w = synth.matrix(fmt, N, K, 7)
    eye = np.eye(K, dtype=np.float32)
    Xb = _bf16_bits_of(eye)
    m = q.Matrix(fmt, N, K, to_dev(w))
    y = _run(m, Xb, K)
    ref = oracle.dequant_rows(fmt, w, N, K).astype(np.float32)
    want = _bf16_bits_of(ref).T  # [K, N]
    got = _bf16_bits_of(y)       # y holds bf16 values exactly; compare as bits
    assert np.array_equal(y, y.astype(np.float32))
    assert np.array_equal(got, want)
    # and y itself is exactly the bf16 value widened to fp32
    widened = (want.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(y.view(np.uint32), widened.view(np.uint32))
    m.close()


@pytest.mark.parametrize("tok", [None, 128, 256])
@pytest.mark.parametrize("M,N,K", [
    (1, 256, 256), (5, 300, 512), (128, 256, 1024), (130, 513, 768), (257, 1024, 2048),
    (300, 64, 256), (129, 257, 4096),
])
def test_gemm_small(monkeypatch, tok, M, N, K):
    """Small and ragged shapes, with the token tile chosen by the library or
    forced to 128 or 256."""
    if tok:
        monkeypatch.setenv("QMM_GEMM_TOK", str(tok))
    _check(M, N, K, seed=M + N + K)


@pytest.mark.parametrize("fmt", [12, 8])
@pytest.mark.parametrize("tok", [128, 256])
def test_gemm_identity_both_tiles(monkeypatch, tok, fmt):
    monkeypatch.setenv("QMM_GEMM_TOK", str(tok))
    test_gemm_identity_is_bf16_weights(fmt)


@pytest.mark.parametrize("tok", [None, 128, 256])
@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (130, 513, 768), (257, 1024, 2048),
                                   (129, 257, 4096)])
def test_gemm_q8_0_small(monkeypatch, tok, M, N, K):
    """Q8_0 weights (two 34-byte blocks per 64-weight step, staged as 80-byte
    windows) on small and ragged shapes."""
    if tok:
        monkeypatch.setenv("QMM_GEMM_TOK", str(tok))
    _check(M, N, K, seed=M + N + K + 8, fmt=q.Q8_0)


@pytest.mark.parametrize("N,K", [(4096, 4096), (4096, 14336)])
def test_gemm_q8_0_llama_shapes_m512(N, K):
    rng = np.random.default_rng(N + K + 8)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N), rng.choice(N, 48, False)]))
    _check(512, N, K, seed=N * 5 + K, rows=rows, fmt=q.Q8_0)


@pytest.mark.parametrize("ksplit", [2, 3, 4])
def test_gemm_q8_0_split_k(monkeypatch, ksplit):
    monkeypatch.setenv("QMM_GEMM_KSPLIT", str(ksplit))
    _check(200, 512, 2048, seed=31, fmt=q.Q8_0)


@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_gemm_llama_shapes_m512(N, K):
    """The Llama-3.1-8B shapes at M = 512 tokens, on sampled rows (every
    token, the first/last row tiles and random rows)."""
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N), rng.choice(N, 48, False)]))
    _check(512, N, K, seed=N * 3 + K, rows=rows)


def test_gemm_m2048_sampled():
    rng = np.random.default_rng(5)
    N, K = 4096, 4096
    rows = np.unique(np.concatenate([np.arange(4), np.arange(N - 4, N), rng.choice(N, 24, False)]))
    _check(2048, N, K, seed=99, rows=rows)


def test_gemm_deterministic_and_graph():
    M, N, K = 384, 1024, 1024
    w = synth.q4k_matrix(N, K, 3)
    Xb = to_dev(synth.activations_bf16(M, K, 4).view(np.int16))
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    Y1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    Y2 = torch.empty_like(Y1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        m.gemm(Xb, Y1, stream=s)
        m.gemm(Xb, Y2, stream=s)
    s.synchronize()
    assert torch.equal(Y1.view(torch.int32), Y2.view(torch.int32))
    g = torch.cuda.CUDAGraph()
    Y3 = torch.zeros_like(Y1)
    with torch.cuda.graph(g, stream=s):
        m.gemm(Xb, Y3, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int32), Y3.view(torch.int32))
    m.close()


def test_gemm_refusals():
    N, K = 64, 256
    w6 = synth.matrix(q.Q6_K, N, K, 1)
    m6 = q.Matrix(q.Q6_K, N, K, to_dev(w6))
    X = torch.zeros((4, K), dtype=torch.int16, device="cuda")
    Y = torch.zeros((4, N), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        m6.gemm(X, Y)
    assert ei.value.status == q.ERR_UNSUPPORTED and "Q4_K" in ei.value.message
    m6.close()
    w8 = synth.matrix(q.Q8_0, N, 96, 1)  # rows not whole 256-weight groups
    m8 = q.Matrix(q.Q8_0, N, 96, to_dev(w8))
    with pytest.raises(q.QmmError) as ei:
        m8.gemm(torch.zeros((4, 96), dtype=torch.int16, device="cuda"), Y)
    assert ei.value.status == q.ERR_UNSUPPORTED
    m8.close()
    w = synth.q4k_matrix(N, K, 2)
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    with pytest.raises(q.QmmError) as ei:
        q.gemm(m.h, X, 0, Y)
    assert ei.value.status == q.ERR_SHAPE
    with pytest.raises(q.QmmError) as ei:
        q.gemm(m.h, X.data_ptr() + 2, 2, Y)
    assert ei.value.status == q.ERR_ALIGN
    with pytest.raises(q.QmmError) as ei:
        q.gemm(m.h, None, 2, Y)
    assert ei.value.status == q.ERR_NULL
    m.close()


@pytest.mark.parametrize("ksplit", [2, 3, 4, 5, 7, 8])
def test_gemm_split_k_forced(monkeypatch, ksplit):
    """K split over several CTAs, the partial products added in slice order by
    a reduction kernel: within bounds, and repeatable bit for bit.  K = 2048
    has 8 super-blocks, so 3, 5 and 7 slices are uneven (super-blocks
    [k * 8 / ks, (k + 1) * 8 / ks) each)."""
    monkeypatch.setenv("QMM_GEMM_KSPLIT", str(ksplit))
    M, N, K = 300, 513, 2048
    y = _check(M, N, K, seed=ksplit)
    w = synth.q4k_matrix(N, K, ksplit)
    Xb = synth.activations_bf16(M, K, ksplit + 1)
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    y2 = _run(m, Xb, M)
    y3 = _run(m, Xb, M)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(y2.view(np.uint32), y3.view(np.uint32))
    m.close()


@pytest.mark.parametrize("ksplit", [None, 2])
@pytest.mark.parametrize("Ns,K,M", [((300, 64, 513), 1024, 300), ((4096, 1024, 1024), 4096, 512)])
def test_gemm_group(monkeypatch, ksplit, Ns, K, M):
    """qmm_gemm_group: matrices sharing X in one launch (ragged row counts, so
    row tiles of different matrices meet mid-launch), each against the oracle."""
    if ksplit:
        monkeypatch.setenv("QMM_GEMM_KSPLIT", str(ksplit))
    ws = [synth.q4k_matrix(N, K, 40 + i) for i, N in enumerate(Ns)]
    ms = [q.Matrix(q.Q4_K, N, K, to_dev(w)) for N, w in zip(Ns, ws)]
    Xb = synth.activations_bf16(M, K, 41)
    Ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
    q.gemm_group([m.h for m in ms], to_dev(Xb.view(np.int16)), M, Ys)
    torch.cuda.synchronize()
    rng = np.random.default_rng(K)
    for N, w, Y in zip(Ns, ws, Ys):
        rows = None if N <= 600 else np.unique(np.concatenate(
            [np.arange(4), np.arange(N - 4, N), rng.choice(N, 24, False)]))
        y_ref, c = oracle.gemm_bf16(w, N, K, Xb, rows=rows, nthreads=NTHREADS)
        got = Y.cpu().numpy() if rows is None else Y.cpu().numpy()[:, rows]
        assert_close_to_oracle(got, y_ref, c, TIGHT, f"group N={N}")
    assert ms[0].status() == 0
    for m in ms:
        m.close()


def test_gemm_group_refusals():
    K = 256
    a = q.Matrix(q.Q4_K, 64, K, to_dev(synth.q4k_matrix(64, K, 1)))
    b = q.Matrix(q.Q4_K, 64, 512, to_dev(synth.q4k_matrix(64, 512, 2)))
    X = torch.zeros((4, K), dtype=torch.int16, device="cuda")
    Y = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.gemm_group([a.h, b.h], X, 4, [Y, Y])
    assert ei.value.status == q.ERR_SHAPE
    with pytest.raises(q.QmmError) as ei:
        q.gemm_group([a.h] * 5, X, 4, [Y] * 5)
    assert ei.value.status == q.ERR_SHAPE
    a.close()
    b.close()


def test_gemm_tail_wave_split():
    """More tiles than SMs: full waves run whole tiles, the tail wave's tiles
    are split in K (reduced in slice order) -- rows from both kinds."""
    M, N, K = 300, 20480, 1024
    w = synth.q4k_matrix(N, K, 77)
    Xb = synth.activations_bf16(M, K, 78)
    m = q.Matrix(q.Q4_K, N, K, to_dev(w))
    Y1 = _run(m, Xb, M)
    Y2 = _run(m, Xb, M)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N), rng.choice(N, 56, False),
                                     np.arange(19456, 19456 + 8)]))
    y_ref, c = oracle.gemm_bf16(w, N, K, Xb, rows=rows, nthreads=NTHREADS)
    assert_close_to_oracle(Y1[:, rows], y_ref, c, TIGHT, "tail split")
    m.close()


@pytest.mark.parametrize("fmt", [12, 8])
@pytest.mark.parametrize("ksplit", [None, 3, 4])
@pytest.mark.parametrize("M,N", [(300, 1024), (512, 300)])
def test_gemm_bulk_store_epilogue_matches_thread_stores(monkeypatch, fmt, ksplit, M, N):
    """The epilogue's bulk tensor stores (32 x 32 chunks through shared
    memory; ragged token tiles clipped by the tensor map, a ragged 32-column
    piece left to the threads) write the same bits as per-thread stores,
    into Y and, with K split, into the partials."""
    if ksplit:
        monkeypatch.setenv("QMM_GEMM_KSPLIT", str(ksplit))
    K = 2048
    w = synth.matrix(fmt, N, K, M + N + fmt)
    Xb = synth.activations_bf16(M, K, 7)
    m = q.Matrix(fmt, N, K, to_dev(w))
    y_bulk = _run(m, Xb, M)
    monkeypatch.setenv("QMM_GEMM_THREAD_STORES", "1")
    y_thr = _run(m, Xb, M)
    assert np.all(np.isfinite(y_bulk))
    assert np.array_equal(y_bulk.view(np.uint32), y_thr.view(np.uint32))
    assert m.status() == 0
    m.close()
