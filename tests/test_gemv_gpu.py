"""GPU parity of the decoder and the decode GEMV against the CPU oracle,
through the C ABI.

Dequantised block values must be bit-exact (fp32 and bf16); GEMV outputs
must satisfy |y - y_ref| <= 1e-4 * sum|w x|.  Sizes span several CTAs, ragged
row tails, split-K, grouped launches and the full Llama-3.1-8B shapes (the
big ones on sampled rows)."""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests import _golden
from tests._util import TOL_FP32, assert_close_to_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("quantized_gguf_dequant_gb300")

FMTS = [q.Q4_K, q.Q8_0]


def _matrix(fmt, N, K, seed):
    w = synth.matrix(fmt, N, K, seed)
    return w, q.Matrix(fmt, N, K, to_dev(w))


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 1024), (64, 4096)])
def test_dequant_bit_exact(fmt, N, K):
    w, m = _matrix(fmt, N, K, seed=N * 7 + K)
    ref = oracle.dequant_rows(fmt, w, N, K)
    got = m.dequantize().cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.astype(np.float32).view(np.uint32))
    gb = m.dequantize_bf16().cpu().numpy().view(np.uint16)
    refb = np.array([oracle.bf16_from_float(v) for v in ref.astype(np.float32).ravel()],
                    np.uint16).reshape(ref.shape)
    assert np.array_equal(gb, refb)
    part = m.dequantize(row0=N // 2, nrows=N - N // 2).cpu().numpy()
    assert np.array_equal(part, got[N // 2:])
    m.close()


def test_dequant_golden_blocks():
    for fmt, name, blk, expect in _golden.blocks():
        K = 256 if fmt == q.Q4_K else 256
        reps = 1 if fmt == q.Q4_K else 8  # Q8_0 rows here hold 8 copies of the block
        row = np.frombuffer(blk * reps, np.uint8)
        m = q.Matrix(fmt, 1, K, to_dev(row))
        got = m.dequantize().cpu().numpy()[0]
        for i, v in expect.items():
            assert got[i] == np.float32(v), (name, i, got[i], v)
        m.close()


# ------------------------------------------------------------------ GEMV

def _check_gemv(fmt, N, K, seed, rows=None, x=None):
    w, m = _matrix(fmt, N, K, seed)
    if x is None:
        x = synth.activations(1, K, seed + 1)[0]
    y = m.gemv(to_dev(x)).cpu().numpy()
    y_ref, c = oracle.gemv(fmt, w, N, K, x, rows=rows, nthreads=oracle.max_threads())
    assert_close_to_oracle(y if rows is None else y[rows], y_ref, c, TOL_FP32,
                           f"gemv fmt={fmt} N={N} K={K}")
    assert m.status() == q.OK
    return m, w, x, y


@pytest.mark.parametrize("small", ["default", "4194304"])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K", [(1, 256), (7, 256), (33, 512), (1023, 1024), (1024, 1024),
                                 (257, 2048), (100, 4096), (300, 3072), (5, 14336)])
def test_gemv_small(monkeypatch, small, fmt, N, K):
    """Small shapes on the default route and with Q4_K matrices up to 4 MiB
    sent to the SIMT kernel (QMM_Q4K_SMALL_BYTES)."""
    if small != "default":
        monkeypatch.setenv("QMM_Q4K_SMALL_BYTES", small)
    m, *_ = _check_gemv(fmt, N, K, seed=N + K)
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ksplit", [2, 4])
def test_gemv_forced_split_k(fmt, ksplit, monkeypatch):
    # split-K lives in the fp32 kernel (Q8_0, and Q4_K when asked for it)
    monkeypatch.setenv("QMM_Q4K_PATH", "simt")
    monkeypatch.setenv("QMM_SPLITK", str(ksplit))
    for N, K in ((37, 2048), (300, 4096)):
        m, *_ = _check_gemv(fmt, N, K, seed=ksplit * 100 + N)
        # repeat: tickets must have been reset
        m2, *_ = _check_gemv(fmt, N, K, seed=ksplit * 100 + N)
        m.close()
        m2.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("name,N,K", list(synth.LLAMA8B_SHAPES))
def test_gemv_llama8b_shapes_sampled_rows(fmt, name, N, K):
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 254)]))
    m, *_ = _check_gemv(fmt, N, K, seed=sum(map(ord, name)), rows=rows)
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_deterministic_and_power_of_two_scaling(fmt):
    N, K = 2048, 4096
    w, m = _matrix(fmt, N, K, seed=5)
    x = to_dev(synth.activations(1, K, 6)[0])
    y1 = m.gemv(x).cpu().numpy()
    y2 = m.gemv(x).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    y4 = m.gemv(x * 4.0).cpu().numpy()
    assert np.array_equal(y4, 4.0 * y1)
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_edge_activations(fmt):
    N, K = 64, 1024
    w, m = _matrix(fmt, N, K, seed=8)
    x0 = np.zeros(K, np.float32)
    y0 = m.gemv(to_dev(x0)).cpu().numpy()
    assert np.all(y0 == 0)
    rng = np.random.default_rng(9)
    # wide dynamic range, tiny and huge magnitudes, one-hot
    cases = [
        (rng.standard_normal(K) * np.exp(rng.uniform(-40, 40, K))).astype(np.float32),
        (rng.standard_normal(K) * 1e-30).astype(np.float32),
        (rng.standard_normal(K) * 1e20).astype(np.float32),
        np.eye(1, K, 777, dtype=np.float32)[0],
    ]
    for x in cases:
        y = m.gemv(to_dev(x)).cpu().numpy()
        y_ref, c = oracle.gemv(fmt, w, N, K, x)
        assert_close_to_oracle(y, y_ref, c, TOL_FP32, f"edge fmt={fmt}")
    # one-hot picks a column exactly (every product exact, one term)
    W = oracle.dequant_rows(fmt, w, N, K)
    y = m.gemv(to_dev(cases[-1])).cpu().numpy()
    assert np.array_equal(y, W[:, 777].astype(np.float32))
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_leaves_neighbours_untouched(fmt):
    N, K = 333, 1024
    w, m = _matrix(fmt, N, K, seed=10)
    x = synth.activations(1, K, 11)[0]
    buf = torch.full((N + 64,), 12345.0, dtype=torch.float32, device="cuda")
    q.gemv(m.h, to_dev(x), buf[32:32 + N])
    out = buf.cpu().numpy()
    assert np.all(out[:32] == 12345.0) and np.all(out[32 + N:] == 12345.0)
    y_ref, c = oracle.gemv(fmt, w, N, K, x)
    assert_close_to_oracle(out[32:32 + N], y_ref, c, TOL_FP32, "canary")
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_group_matches_separate(fmt):
    K = 4096
    shapes = [(4096, K), (1024, K), (1024, K)]
    mats, ws = [], []
    for i, (N, _) in enumerate(shapes):
        w, m = _matrix(fmt, N, K, seed=40 + i)
        mats.append(m)
        ws.append(w)
    x = synth.activations(1, K, 44)[0]
    xd = to_dev(x)
    ys = [torch.empty(N, dtype=torch.float32, device="cuda") for N, _ in shapes]
    q.gemv_group([m.h for m in mats], xd, ys)
    for m, w, y, (N, _) in zip(mats, ws, ys, shapes):
        y_ref, c = oracle.gemv(fmt, w, N, K, x, nthreads=oracle.max_threads())
        assert_close_to_oracle(y.cpu().numpy(), y_ref, c, TOL_FP32, "group")
        ys_sep = m.gemv(xd).cpu().numpy()
        assert np.all(np.isfinite(ys_sep))
    for m in mats:
        m.close()


def test_gemv_refusals_on_device():
    w, m = _matrix(q.Q4_K, 16, 256, seed=1)
    x = torch.zeros(260, dtype=torch.float32, device="cuda")
    y = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.gemv(m.h, x[1:], y)
    assert e.value.status == q.ERR_ALIGN and "x is not 16-byte aligned" in e.value.message
    w8, m8 = _matrix(q.Q8_0, 16, 512, seed=2)
    with pytest.raises(q.QmmError) as e:
        q.gemv_group([m.h, m8.h], x, [y, y])
    assert e.value.status == q.ERR_SHAPE and "differs from matrix 0" in e.value.message
    m.close()
    m8.close()


@pytest.mark.parametrize("N,K", [(1, 256), (17, 512), (1000, 4096), (4096, 1024), (300, 14336)])
def test_gemv_q4k_fp32_kernel(N, K, monkeypatch):
    """The fp32 (SIMT) Q4_K kernel, kept for K whose activations exceed the
    tensor-core kernel's shared memory."""
    monkeypatch.setenv("QMM_Q4K_PATH", "simt")
    m, *_ = _check_gemv(q.Q4_K, N, K, seed=N * 3 + K)
    m.close()


@pytest.mark.parametrize("S", ["1", "2", "4", "7", "8", "16"])
def test_gemv_m1_forced_k_slices(S, monkeypatch):
    """The one-row decode kernel with every K-slice count that divides the
    shape's super-blocks (others fall back to the default plan): ragged row
    tiles, slot groups of one to eight tiles, row segments of one to eight
    super-blocks, slices added by the last CTA; twice, so the row-group
    tickets must have been reset."""
    monkeypatch.setenv("QMM_M1_S", S)
    monkeypatch.setenv("QMM_Q4K_SMALL_BYTES", "0")  # the decode kernel even for small shapes
    for N, K in ((37, 2048), (300, 4096), (1000, 1024), (77, 14336), (1, 256), (40, 768),
                 (4096, 3584)):
        for rep in range(2):
            m, *_ = _check_gemv(q.Q4_K, N, K, seed=int(S) * 1000 + N + rep)
            m.close()


@pytest.mark.parametrize("S", ["1", "4"])
def test_gemv_m1_ragged_group(S, monkeypatch):
    """A group of matrices with ragged row counts sharing x: slots that
    straddle two matrices, rows past a matrix end never written."""
    monkeypatch.setenv("QMM_M1_S", S)
    monkeypatch.setenv("QMM_Q4K_SMALL_BYTES", "0")
    K = 2048
    shapes = [17, 1, 250, 33]
    mats, ws = [], []
    for i, N in enumerate(shapes):
        w, m = _matrix(q.Q4_K, N, K, seed=70 + i)
        mats.append(m)
        ws.append(w)
    x = synth.activations(1, K, 74)[0]
    bufs = [torch.full((N + 8,), 777.0, dtype=torch.float32, device="cuda") for N in shapes]
    q.gemv_group([m.h for m in mats], to_dev(x), [b[4:4 + N] for b, N in zip(bufs, shapes)])
    for w, b, N in zip(ws, bufs, shapes):
        out = b.cpu().numpy()
        assert np.all(out[:4] == 777.0) and np.all(out[4 + N:] == 777.0)
        y_ref, c = oracle.gemv(q.Q4_K, w, N, K, x)
        assert_close_to_oracle(out[4:4 + N], y_ref, c, TOL_FP32, f"ragged group N={N}")
    for m in mats:
        m.close()


@pytest.mark.parametrize("nslot,warps", [("2", "8"), ("3", "16"), ("6", "8"), ("4", "12")])
def test_gemv_q4k_tensor_core_shapes(nslot, warps, monkeypatch):
    """The tensor-core kernel with other ring depths / CTA sizes, and on a
    long K where the fp32 kernel would normally be chosen."""
    monkeypatch.setenv("QMM_Q4K_PATH", "tc")
    monkeypatch.setenv("QMM_TC_NSLOT", nslot)
    monkeypatch.setenv("QMM_TC_WARPS", warps)
    for N, K in ((2048, 4096), (77, 14336), (1, 256), (40, 768)):
        m, *_ = _check_gemv(q.Q4_K, N, K, seed=int(nslot) * 10 + N)
        m.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 16])
def test_gemv_batched(fmt, M):
    N, K = 1000, 4096
    w, m = _matrix(fmt, N, K, seed=70 + M)
    X = synth.activations(M, K, seed=71 + M)
    Y = m.gemv_batched(to_dev(X)).cpu().numpy()
    Yr, C = oracle.gemv(fmt, w, N, K, X, nthreads=oracle.max_threads())
    assert_close_to_oracle(Y, Yr, C, TOL_FP32, f"batched fmt={fmt} M={M}")
    # row m of the batch equals the single-vector GEMV of row m
    for r in (0, M - 1):
        y1 = m.gemv(to_dev(X[r])).cpu().numpy()
        assert_close_to_oracle(y1, Yr[r], C[r], TOL_FP32, "batched row")
    m.close()


def test_gemv_batched_strided_and_big_k():
    N, K, M = 333, 14336, 4
    w, m = _matrix(q.Q4_K, N, K, seed=90)
    X = synth.activations(M, K + 64, seed=91)  # ldx = K + 64
    Xd = to_dev(X)
    Yd = torch.full((M, N + 8), 7.0, dtype=torch.float32, device="cuda")
    q.gemv_batched(m.h, Xd, M, K + 64, Yd, N + 8)
    Y = Yd.cpu().numpy()
    assert np.all(Y[:, N:] == 7.0)
    Yr, C = oracle.gemv(q.Q4_K, w, N, K, np.ascontiguousarray(X[:, :K]),
                        nthreads=oracle.max_threads())
    assert_close_to_oracle(Y[:, :N], Yr, C, TOL_FP32, "batched strided")
    m.close()


@pytest.mark.parametrize("M", [2, 5, 8, 12, 16])
@pytest.mark.parametrize("N,K", [(4096, 14336), (1024, 4096), (300, 768)])
def test_gemv_batched_one_pass(M, N, K):
    """All M rows in one pass (K sliced across CTAs where needed), against
    the oracle on sampled rows of the large shapes."""
    w, m = _matrix(q.Q4_K, N, K, seed=M * 11 + K)
    X = synth.activations(M, K, seed=M + N)
    Y = m.gemv_batched(to_dev(X)).cpu().numpy()
    rng = np.random.default_rng(M)
    rows = None if N <= 1024 else np.unique(np.concatenate(
        [np.arange(16), np.arange(N - 16, N), rng.choice(N, 64, False)]))
    Yr, C = oracle.gemv(q.Q4_K, w, N, K, X, rows=rows, nthreads=oracle.max_threads())
    got = Y if rows is None else Y[:, rows]
    assert_close_to_oracle(got, Yr, C, TOL_FP32, f"batched one pass M={M} N={N} K={K}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("M", [2, 3, 8, 9, 16])
@pytest.mark.parametrize("N,K", [(300, 768), (257, 2048), (1024, 4096), (4096, 14336)])
def test_gemv_batched_tc5(monkeypatch, M, N, K):
    """The tcgen05 batched decode (QMM_BATCHED_PATH=tc5: 256-row tiles, K
    slices chosen by the planner, 16 or 32 B columns) against the oracle;
    large shapes on sampled rows."""
    monkeypatch.setenv("QMM_BATCHED_PATH", "tc5")
    w, m = _matrix(q.Q4_K, N, K, seed=M * 7 + N + K)
    X = synth.activations(M, K, seed=M + 3 * N)
    Y = m.gemv_batched(to_dev(X)).cpu().numpy()
    rng = np.random.default_rng(M + N)
    rows = None if N <= 1024 else np.unique(np.concatenate(
        [np.arange(16), np.arange(N - 16, N), rng.choice(N, 96, False)]))
    Yr, C = oracle.gemv(q.Q4_K, w, N, K, X, rows=rows, nthreads=oracle.max_threads())
    got = Y if rows is None else Y[:, rows]
    assert_close_to_oracle(got, Yr, C, TOL_FP32, f"tc5 M={M} N={N} K={K}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("S", [1, 2, 3, 7, 14])
@pytest.mark.parametrize("M", [9, 16])
def test_gemv_batched_tc5_forced_slices(monkeypatch, S, M):
    """K slices whose partial sums the last slice of each (tile, warp) adds
    in slice order: within bounds, bitwise repeatable, tickets left at zero
    (a second call gives the same bits)."""
    monkeypatch.setenv("QMM_BATCHED_PATH", "tc5")
    monkeypatch.setenv("QMM_TC5_S", str(S))
    N, K = 515, 256 * 14
    w, m = _matrix(q.Q4_K, N, K, seed=S + M)
    X = synth.activations(M, K, seed=S + 1)
    Y1 = m.gemv_batched(to_dev(X)).cpu().numpy()
    Y2 = m.gemv_batched(to_dev(X)).cpu().numpy()
    Yr, C = oracle.gemv(q.Q4_K, w, N, K, X, nthreads=oracle.max_threads())
    assert_close_to_oracle(Y1, Yr, C, TOL_FP32, f"tc5 S={S} M={M}")
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    m.close()


@pytest.mark.parametrize("path", ["tc5", "tcb"])
def test_gemv_batched_edge_activations(monkeypatch, path):
    """Rows of very different magnitudes (the per-token, per-super-block
    power-of-two scale), an all-zero row and a row with one nonzero value,
    on both batched kernels."""
    monkeypatch.setenv("QMM_BATCHED_PATH", path)
    N, K, M = 384, 1024, 6
    w, m = _matrix(q.Q4_K, N, K, seed=44)
    X = synth.activations(M, K, seed=45)
    X[0] *= np.float32(1e30)
    X[1] *= np.float32(1e-30)
    X[2] = 0.0
    X[3] = 0.0
    X[3, 517] = 3.0
    X[4, :256] *= np.float32(1e20)  # one super-block far larger than the rest
    Y = m.gemv_batched(to_dev(X)).cpu().numpy()
    Yr, C = oracle.gemv(q.Q4_K, w, N, K, X, nthreads=oracle.max_threads())
    assert_close_to_oracle(Y, Yr, C, TOL_FP32, f"{path} edge activations")
    assert np.all(Y[2] == 0.0)
    m.close()


@pytest.mark.parametrize("S", [2, 3, 7])
def test_gemv_batched_forced_k_slices(monkeypatch, S):
    """The mma.sync batched kernel (QMM_BATCHED_PATH=tcb): K split into S
    slices whose partial sums a reduction kernel adds in slice order: within
    bounds and bitwise repeatable."""
    monkeypatch.setenv("QMM_BATCHED_PATH", "tcb")
    monkeypatch.setenv("QMM_TCB_S", str(S))
    N, K, M = 515, 256 * 14, 9
    w, m = _matrix(q.Q4_K, N, K, seed=S)
    X = synth.activations(M, K, seed=S + 1)
    Y1 = m.gemv_batched(to_dev(X)).cpu().numpy()
    Y2 = m.gemv_batched(to_dev(X)).cpu().numpy()
    Yr, C = oracle.gemv(q.Q4_K, w, N, K, X, nthreads=oracle.max_threads())
    assert_close_to_oracle(Y1, Yr, C, TOL_FP32, f"batched S={S}")
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    m.close()


@pytest.mark.parametrize("path", ["default", "staged"])
@pytest.mark.parametrize("N,K", [(1, 256), (33, 768), (300, 2048), (1000, 4096), (77, 14336),
                                 (4096, 14336)])
def test_q8_0_routes(monkeypatch, path, N, K):
    """Q8_0 on the tensor-core decode kernel (the default where K is a
    multiple of 256) and on the staged fp32 kernel (QMM_FMT_PATH=staged),
    sampled rows at the largest shape; grouped launch of two matrices too."""
    if path != "default":
        monkeypatch.setenv("QMM_FMT_PATH", path)
    rng = np.random.default_rng(N + K)
    rows = None if N <= 1000 else np.unique(np.concatenate(
        [np.arange(16), np.arange(N - 16, N), rng.choice(N, 64, False)]))
    m, w, x, y = _check_gemv(q.Q8_0, N, K, seed=N * 3 + K, rows=rows)
    w2, m2 = _matrix(q.Q8_0, 40, K, seed=N + 1)
    y1 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    y2 = torch.full((40,), float("nan"), dtype=torch.float32, device="cuda")
    q.gemv_group([m.h, m2.h], to_dev(x), [y1, y2])
    torch.cuda.synchronize()
    yr1, c1 = oracle.gemv(q.Q8_0, w, N, K, x, rows=rows, nthreads=oracle.max_threads())
    y1h = y1.cpu().numpy()
    assert_close_to_oracle(y1h if rows is None else y1h[rows], yr1, c1, TOL_FP32, "group 0")
    yr2, c2 = oracle.gemv(q.Q8_0, w2, 40, K, x, nthreads=oracle.max_threads())
    assert_close_to_oracle(y2.cpu().numpy(), yr2, c2, TOL_FP32, "group 1")
    m.close()
    m2.close()


def test_launch_count_counts_kernels():
    """qmm_launch_count advances by the kernels each call launches."""
    w, m = _matrix(q.Q4_K, 512, 1024, seed=5)
    x = to_dev(synth.activations(1, 1024, 6)[0])
    c0 = q.launch_count()
    m.gemv(x)
    torch.cuda.synchronize()
    assert q.launch_count() - c0 == 1
    m.close()
    # K in slices: for one or four rows the slices are added inside the same
    # launch (last CTA of each row group); for sixteen rows by a second kernel.
    w, m = _matrix(q.Q4_K, 512, 14336, seed=7)
    x = to_dev(synth.activations(16, 14336, 8))
    c0 = q.launch_count()
    m.gemv(x[0])
    m.gemv_batched(x[:4])
    torch.cuda.synchronize()
    assert q.launch_count() - c0 == 2
    c0 = q.launch_count()
    m.gemv_batched(x)
    torch.cuda.synchronize()
    assert q.launch_count() - c0 == 2
    m.close()


def test_gemv_chain_in_cuda_graph_matches_eager():
    """Launch chaining: a grouped q/k/v call, a single call and the long-K
    call captured in one CUDA graph (programmatic dependent launch between
    them) replay to the same bits as eager launches."""
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096), (512, 4096), (1024, 14336)]
    mats, ws = [], []
    for i, (N, K) in enumerate(shapes):
        w, m = _matrix(q.Q4_K, N, K, seed=300 + i)
        mats.append(m)
        ws.append(w)
    x1 = to_dev(synth.activations(1, 4096, 301)[0])
    x2 = to_dev(synth.activations(1, 14336, 302)[0])
    ys = [torch.zeros(N, dtype=torch.float32, device="cuda") for N, _ in shapes]

    def step(stream):
        q.gemv_group([mats[0].h, mats[1].h, mats[2].h], x1, ys[0:3], stream)
        q.gemv(mats[3].h, x1, ys[3], stream)
        q.gemv(mats[4].h, x2, ys[4], stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    s.synchronize()
    eager = [y.clone() for y in ys]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for y in ys:
        y.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ys, eager):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    y_ref, c = oracle.gemv(q.Q4_K, ws[4], 1024, 14336, x2.cpu().numpy(), nthreads=oracle.max_threads())
    assert_close_to_oracle(ys[4].cpu().numpy(), np.ravel(y_ref), np.ravel(c), TOL_FP32, "chain long K")
    for m in mats:
        m.close()


@pytest.mark.parametrize("N,K", [(1, 256), (37, 2048), (1024, 1024), (300, 4096), (77, 14336),
                                 (5, 8192), (33, 768)])
def test_gemv_q4k_simt_small_shape_path(monkeypatch, N, K):
    """The SIMT decode kernel for Q4_K (the small-shape path; forced here with
    QMM_Q4K_PATH=fmt): one matrix and a group, against the oracle."""
    monkeypatch.setenv("QMM_Q4K_PATH", "fmt")
    w, m = _matrix(q.Q4_K, N, K, seed=N + 2 * K)
    x = synth.activations(1, K, seed=N + 1)[0]
    y = m.gemv(to_dev(x)).cpu().numpy()
    yr, c = oracle.gemv(q.Q4_K, w, N, K, x, nthreads=oracle.max_threads())
    assert_close_to_oracle(y, yr, c, TOL_FP32, f"q4k simt N={N} K={K}")
    w2, m2 = _matrix(q.Q4_K, 19, K, seed=N + 3)
    ys = [torch.full((N,), float("nan"), device="cuda"), torch.full((19,), float("nan"), device="cuda")]
    q.gemv_group([m.h, m2.h], to_dev(x), ys)
    torch.cuda.synchronize()
    assert_close_to_oracle(ys[0].cpu().numpy(), yr, c, TOL_FP32, "group 0")
    yr2, c2 = oracle.gemv(q.Q4_K, w2, 19, K, x, nthreads=oracle.max_threads())
    assert_close_to_oracle(ys[1].cpu().numpy(), yr2, c2, TOL_FP32, "group 1")
    m.close()
    m2.close()
