"""GPU parity of the mixture-of-experts path (bucketing by router ids, the
grouped expert GEMV, SwiGLU, the routing-weighted combine and the whole
expert FFN) against the CPU oracle, through the C ABI.

Per-slot and combined outputs must satisfy |y - y_ref| <= 1e-4 * C with C
the oracle's sum of |w x| (times |r| when combined).  For the whole FFN the
bound carries the gate/up bounds through SwiGLU into the down projection
(first order; |silu'| <= 1.1)."""
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

NTHREADS = max(1, oracle.max_threads())


FMTS = [q.Q4_K, q.Q8_0]


def _stacked(E, Ne, K, seed, fmt=q.Q4_K):
    w = synth.matrix(fmt, E * Ne, K, seed)
    return w, q.Matrix(fmt, E * Ne, K, to_dev(w))


def _ids_uniform(T, E, top_k, seed):
    ids, r = synth.router(T, E, top_k, seed)
    return ids, r


def _run_moe(m, E, ids, X, x_per_slot, r=None):
    T, top_k = ids.shape
    Ne = m.N // E
    rows = T if r is not None else T * top_k
    Y = torch.full((rows, Ne), float("nan"), dtype=torch.float32, device="cuda")
    q.moe_gemv(m.h, E, to_dev(ids), T, top_k, to_dev(X), x_per_slot,
               None if r is None else to_dev(r), Y)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


# ------------------------------------------------------------------ SwiGLU

@pytest.mark.parametrize("n", [1, 7, 1000, 1 << 20])
def test_swiglu(n):
    rng = np.random.default_rng(n)
    g = (rng.standard_normal(n) * 6).astype(np.float32)
    u = rng.standard_normal(n).astype(np.float32)
    if n >= 7:
        g[:6] = [0.0, -0.0, 88.0, -88.0, 1e-30, -120.0]
    ref = oracle.swiglu(g, u)
    h = torch.empty(n, dtype=torch.float32, device="cuda")
    q.swiglu(to_dev(g), to_dev(u), h, n)
    got = h.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(ref) + 1e-37)


def test_swiglu_empty():
    h = torch.empty(4, dtype=torch.float32, device="cuda")
    q.swiglu(h, h, h, 0)


# ------------------------------------------------------------------ expert GEMV

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("E,Ne,K,T,top_k,x_per_slot,routed", [
    (8, 48, 512, 5, 3, False, False),     # rows per expert not a multiple of 16
    (4, 40, 256, 16, 2, True, True),
    (16, 64, 1024, 9, 4, False, True),
    (3, 1000, 768, 2, 3, True, False),    # every expert, ragged tiles
    (5, 100, 4096, 7, 5, True, True),     # 16 K-slices per row
])
def test_moe_gemv_small(fmt, E, Ne, K, T, top_k, x_per_slot, routed):
    w, m = _stacked(E, Ne, K, seed=E * 31 + K, fmt=fmt)
    ids, r = _ids_uniform(T, E, top_k, seed=T * 7 + E)
    X = synth.activations(T * top_k if x_per_slot else T, K, seed=K + T)
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, x_per_slot,
                               r if routed else None, nthreads=NTHREADS)
    y = _run_moe(m, E, ids, X, x_per_slot, r if routed else None)
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, f"moe E={E} Ne={Ne} K={K}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("which", ["gate", "down"])
def test_moe_gemv_olmoe(fmt, which):
    """The OLMoE expert shapes: 64 experts, d_model 2048, d_ff 1024, 32
    tokens, top-8 (gate: per-slot outputs from shared token inputs; down:
    per-slot inputs, routing-weighted sum)."""
    E, T, top_k = synth.OLMOE_EXPERTS, 32, synth.OLMOE_TOP_K
    if which == "gate":
        Ne, K, xps, routed = synth.OLMOE_D_FF, synth.OLMOE_D_MODEL, False, False
    else:
        Ne, K, xps, routed = synth.OLMOE_D_MODEL, synth.OLMOE_D_FF, True, True
    w, m = _stacked(E, Ne, K, seed=11 if which == "gate" else 12, fmt=fmt)
    ids, r = _ids_uniform(T, E, top_k, seed=5)
    X = synth.activations(T * top_k if xps else T, K, seed=6)
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, xps, r if routed else None,
                               nthreads=NTHREADS)
    y = _run_moe(m, E, ids, X, xps, r if routed else None)
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, f"olmoe {which}")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_moe_gemv_one_hot_expert(fmt):
    """Every slot routed to one expert: that expert's slots form many groups."""
    E, Ne, K, T = 16, 64, 512, 41
    w, m = _stacked(E, Ne, K, seed=3, fmt=fmt)
    ids = np.full((T, 1), 5, np.int32)
    X = synth.activations(T, K, seed=4)
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, False, nthreads=NTHREADS)
    y = _run_moe(m, E, ids, X, False)
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, "one expert")
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_moe_gemv_repeated_expert_in_token(fmt):
    """ids need not be distinct within a token."""
    E, Ne, K, T, top_k = 4, 32, 256, 6, 4
    w, m = _stacked(E, Ne, K, seed=8, fmt=fmt)
    ids = np.array([[1, 1, 2, 1]] * T, np.int32)
    r = np.full((T, top_k), 0.25, np.float32)
    X = synth.activations(T, K, seed=9)
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, False, r, nthreads=NTHREADS)
    y = _run_moe(m, E, ids, X, False, r)
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, "repeated ids")
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("routed", [False, True])
def test_moe_gemv_bad_ids(fmt, routed):
    """Ids outside [0, E): the slot contributes 0, the status word says so."""
    E, Ne, K, T, top_k = 8, 32, 256, 6, 2
    w, m = _stacked(E, Ne, K, seed=21, fmt=fmt)
    ids, r = _ids_uniform(T, E, top_k, seed=22)
    bad = [(1, 0), (4, 1)]
    ids_bad = ids.copy()
    ids_bad[1, 0] = E
    ids_bad[4, 1] = -3
    X = synth.activations(T, K, seed=23)
    r_use = r.copy()
    for t, s in bad:
        r_use[t, s] = 0.0
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, False,
                               r_use if routed else None, nthreads=NTHREADS)
    if not routed:
        for t, s in bad:
            y_ref[t * top_k + s] = 0.0
            c[t * top_k + s] = 0.0
    y = _run_moe(m, E, ids_bad, X, False, r if routed else None)
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, "bad ids")
    if not routed:
        for t, s in bad:
            assert np.all(y[t * top_k + s] == 0.0)
    assert m.status() == q.ERR_EXPERT
    assert m.status() == 0  # reading the status clears it
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_moe_gemv_edge_activations(fmt):
    """Token rows of very different magnitudes (the per-block power-of-two
    scale of the activations), an all-zero row and a one-hot row."""
    E, Ne, K, T, top_k = 4, 64, 512, 6, 2
    w, m = _stacked(E, Ne, K, seed=61, fmt=fmt)
    ids = np.array([[0, 1], [0, 2], [1, 3], [0, 3], [2, 1], [3, 0]], np.int32)
    X = synth.activations(T, K, seed=62)
    X[0] *= np.float32(1e30)
    X[1] *= np.float32(1e-30)
    X[2] = 0.0
    X[3] = 0.0
    X[3, 300] = 2.5
    X[4, :32] *= np.float32(1e20)  # one block far larger than the rest
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, False, nthreads=NTHREADS)
    y = _run_moe(m, E, ids, X, False)
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, f"moe edge activations fmt={fmt}")
    assert np.all(y[4:6] == 0.0)  # token 2's slots
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_moe_gemv_deterministic(fmt):
    E, Ne, K, T, top_k = 64, 128, 1024, 32, 8
    w, m = _stacked(E, Ne, K, seed=31, fmt=fmt)
    ids, r = _ids_uniform(T, E, top_k, seed=32)
    X = synth.activations(T, K, seed=33)
    a = _run_moe(m, E, ids, X, False, r)
    b = _run_moe(m, E, ids, X, False, r)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    m.close()


def test_moe_gemv_refusals():
    E, Ne, K = 4, 32, 256
    w, m = _stacked(E, Ne, K, seed=1)
    ids = to_dev(np.zeros((2, 2), np.int32))
    X = torch.zeros((4, K), dtype=torch.float32, device="cuda")
    Y = torch.zeros((4, Ne), dtype=torch.float32, device="cuda")
    cases = [
        (dict(n_experts=3), q.ERR_SHAPE),              # 128 rows do not split into 3
        (dict(top_k=17, T=1), q.ERR_SHAPE),
        (dict(T=4097, top_k=1), q.ERR_SHAPE),
        (dict(T=0), q.ERR_SHAPE),
        (dict(ids=None), q.ERR_NULL),
        (dict(x_per_slot=2), q.ERR_SHAPE),
        (dict(n_experts=0), q.ERR_SHAPE),
    ]
    for kw, code in cases:
        a = dict(n_experts=E, ids=ids, T=2, top_k=2, x_per_slot=0)
        a.update(kw)
        with pytest.raises(q.QmmError) as ei:
            q.moe_gemv(m.h, a["n_experts"], a["ids"], a["T"], a["top_k"], X, a["x_per_slot"],
                       None, Y)
        assert ei.value.status == code, (kw, ei.value)
    m.close()
    # Q8_0 rows whose K is not a multiple of 256 (2-byte aligned only)
    K8 = 288
    w8 = synth.q8_0_matrix(E * Ne, K8, 2)
    m8 = q.Matrix(q.Q8_0, E * Ne, K8, to_dev(w8))
    X8 = torch.zeros((4, K8), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.moe_gemv(m8.h, E, ids, 2, 2, X8, False, None, Y)
    assert ei.value.status == q.ERR_UNSUPPORTED and "256" in ei.value.message
    m8.close()


# ------------------------------------------------------------------ whole FFN

def _ffn_case(E, d_model, d_ff, T, top_k, seed, fmt=q.Q4_K, fmt_down=None):
    fmt_down = fmt if fmt_down is None else fmt_down
    wg = synth.matrix(fmt, E * d_ff, d_model, seed)
    wu = synth.matrix(fmt, E * d_ff, d_model, seed + 1)
    wd = synth.matrix(fmt_down, E * d_model, d_ff, seed + 2)
    ids, r = synth.router(T, E, top_k, seed + 3)
    X = synth.activations(T, d_model, seed + 4)
    return wg, wu, wd, ids, r, X


def _ffn_bound(wg, wu, wd, E, d_model, d_ff, ids, r, X, fmt=q.Q4_K, fmt_down=None):
    """Reference y and the first-order bound C with |y - y_ref| <= 1e-4 C."""
    fmt_down = fmt if fmt_down is None else fmt_down
    g, cg = oracle.moe_gemv(fmt, wg, E, d_ff, d_model, ids, X, False, nthreads=NTHREADS)
    u, cu = oracle.moe_gemv(fmt, wu, E, d_ff, d_model, ids, X, False, nthreads=NTHREADS)
    h = oracle.swiglu(g, u)
    sg = oracle.swiglu(g, np.ones_like(g))  # silu(g)
    a = np.abs(h) + 1.1 * np.abs(u) * cg + np.abs(sg) * cu
    _, c = oracle.moe_gemv(fmt_down, wd, E, d_model, d_ff, ids, a.astype(np.float32), True,
                           np.abs(r), nthreads=NTHREADS)
    if fmt_down == fmt:
        y = oracle.moe_ffn(fmt, wg, wu, wd, E, d_model, d_ff, ids, X, r, nthreads=NTHREADS)
    else:  # the same composition, with the down projection in its own format
        y, _ = oracle.moe_gemv(fmt_down, wd, E, d_model, d_ff, ids, h.astype(np.float32), True,
                               r, nthreads=NTHREADS)
    return y, c * 1.0001


def _run_ffn(hs, E, ids, r, X, d_model, stream=None):
    T, top_k = ids.shape
    Y = torch.full((T, d_model), float("nan"), dtype=torch.float32, device="cuda")
    q.moe_ffn(hs[0].h, hs[1].h, hs[2].h, E, to_dev(ids), T, top_k, to_dev(X), to_dev(r), Y,
              stream)
    torch.cuda.synchronize()
    return Y


@pytest.mark.parametrize("fmts", [(q.Q4_K, q.Q4_K), (q.Q8_0, q.Q8_0), (q.Q8_0, q.Q4_K)])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("E,d_model,d_ff,T,top_k", [
    (4, 512, 256, 3, 2),
    (6, 768, 512, 9, 3),
    (synth.OLMOE_EXPERTS, synth.OLMOE_D_MODEL, synth.OLMOE_D_FF, 32, synth.OLMOE_TOP_K),
])
def test_moe_ffn(monkeypatch, fmts, fused, E, d_model, d_ff, T, top_k):
    """The whole expert FFN, with SwiGLU fused into the gate/up launch or as
    its own kernel; Q4_K, Q8_0, and Q8_0 gate/up with a Q4_K down."""
    if not fused:
        monkeypatch.setenv("QMM_MOE_NOFUSE", "1")
    fmt, fmt_down = fmts
    wg, wu, wd, ids, r, X = _ffn_case(E, d_model, d_ff, T, top_k, seed=E + T, fmt=fmt,
                                      fmt_down=fmt_down)
    y_ref, c = _ffn_bound(wg, wu, wd, E, d_model, d_ff, ids, r, X, fmt, fmt_down)
    hs = [q.Matrix(fmt, E * d_ff, d_model, to_dev(wg)),
          q.Matrix(fmt, E * d_ff, d_model, to_dev(wu)),
          q.Matrix(fmt_down, E * d_model, d_ff, to_dev(wd))]
    y = _run_ffn(hs, E, ids, r, X, d_model).cpu().numpy()
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, f"ffn E={E}")
    assert hs[0].status() == 0
    for h in hs:
        h.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_moe_ffn_graph_replay(fmt):
    """Captured into a CUDA graph after one eager call, the FFN replays to the
    same bits."""
    E, d_model, d_ff, T, top_k = 8, 512, 256, 4, 2
    wg, wu, wd, ids, r, X = _ffn_case(E, d_model, d_ff, T, top_k, seed=77, fmt=fmt)
    hs = [q.Matrix(fmt, E * d_ff, d_model, to_dev(wg)),
          q.Matrix(fmt, E * d_ff, d_model, to_dev(wu)),
          q.Matrix(fmt, E * d_model, d_ff, to_dev(wd))]
    ids_d, r_d, X_d = to_dev(ids), to_dev(r), to_dev(X)
    Y = torch.zeros((T, d_model), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q.moe_ffn(hs[0].h, hs[1].h, hs[2].h, E, ids_d, T, top_k, X_d, r_d, Y, s)
    s.synchronize()
    eager = Y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q.moe_ffn(hs[0].h, hs[1].h, hs[2].h, E, ids_d, T, top_k, X_d, r_d, Y, s)
    Y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int32), eager.view(torch.int32))
    for h in hs:
        h.close()


def test_moe_ffn_refusals():
    E, d_model, d_ff = 4, 512, 256
    wg, wu, wd, ids, r, X = _ffn_case(E, d_model, d_ff, 2, 2, seed=1)
    hg = q.Matrix(q.Q4_K, E * d_ff, d_model, to_dev(wg))
    hu = q.Matrix(q.Q4_K, E * d_ff, d_model, to_dev(wu))
    hd_wrong = q.Matrix(q.Q4_K, E * d_ff, d_model, to_dev(wu))  # not d_model x d_ff
    Y = torch.zeros((2, d_model), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.moe_ffn(hg.h, hu.h, hd_wrong.h, E, to_dev(ids), 2, 2, to_dev(X), to_dev(r), Y)
    assert ei.value.status == q.ERR_SHAPE
    with pytest.raises(q.QmmError) as ei:
        q.moe_ffn(hg.h, hu.h, hd_wrong.h, E, to_dev(ids), 2, 2, to_dev(X), None, Y)
    assert ei.value.status in (q.ERR_NULL, q.ERR_SHAPE)
    for h in (hg, hu, hd_wrong):
        h.close()
    # gate and up in different formats
    wu8 = synth.q8_0_matrix(E * d_ff, d_model, 3)
    hu8 = q.Matrix(q.Q8_0, E * d_ff, d_model, to_dev(wu8))
    hd = q.Matrix(q.Q4_K, E * d_model, d_ff, to_dev(wd))
    hg = q.Matrix(q.Q4_K, E * d_ff, d_model, to_dev(wg))
    with pytest.raises(q.QmmError) as ei:
        q.moe_ffn(hg.h, hu8.h, hd.h, E, to_dev(ids), 2, 2, to_dev(X), to_dev(r), Y)
    assert ei.value.status == q.ERR_FORMAT
    for h in (hg, hu8, hd):
        h.close()


# ------------------------------------------------------------------ routing on the input (Llama 4)

def _ffn_bound_input(wg, wu, wd, E, d_model, d_ff, ids, r, X, fmt=q.Q4_K):
    """As _ffn_bound, for the routing weight applied to the expert input:
    the gate/up bounds are those of the scaled inputs r x, and the slots are
    summed without r."""
    g, cg = oracle.moe_gemv(fmt, wg, E, d_ff, d_model, ids, X, False, r, nthreads=NTHREADS,
                            route_on_input=True)
    u, cu = oracle.moe_gemv(fmt, wu, E, d_ff, d_model, ids, X, False, r, nthreads=NTHREADS,
                            route_on_input=True)
    h = oracle.swiglu(g, u)
    sg = oracle.swiglu(g, np.ones_like(g))
    a = np.abs(h) + 1.1 * np.abs(u) * cg + np.abs(sg) * cu
    _, c = oracle.moe_gemv(fmt, wd, E, d_model, d_ff, ids, a.astype(np.float32), True,
                           np.ones_like(r), nthreads=NTHREADS)
    y = oracle.moe_ffn(fmt, wg, wu, wd, E, d_model, d_ff, ids, X, r, nthreads=NTHREADS,
                       route_on_input=True)
    return y, c * 1.0001


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("E,Ne,K,T,top_k,x_per_slot", [
    (8, 48, 512, 5, 3, False),
    (4, 40, 256, 16, 2, True),
    (16, 64, 1024, 1, 1, False),   # Llama 4 routes each token to one expert
])
def test_moe_gemv_route_on_input(fmt, E, Ne, K, T, top_k, x_per_slot):
    """Per-slot outputs of the experts on their routing-weighted inputs."""
    w, m = _stacked(E, Ne, K, seed=300 + E, fmt=fmt)
    ids, r = _ids_uniform(T, E, top_k, seed=301 + T)
    r = (r * np.float32(3.0) - np.float32(1.0)).astype(np.float32)  # signs and |r| > 1 too
    X = synth.activations(T * top_k if x_per_slot else T, K, seed=302)
    y_ref, c = oracle.moe_gemv(fmt, w, E, Ne, K, ids, X, x_per_slot, r, nthreads=NTHREADS,
                               route_on_input=True)
    Y = torch.full((T * top_k, Ne), float("nan"), dtype=torch.float32, device="cuda")
    q.moe_gemv(m.h, E, to_dev(ids), T, top_k, to_dev(X), x_per_slot, to_dev(r), Y,
               route_on_input=True)
    torch.cuda.synchronize()
    assert_close_to_oracle(Y.cpu().numpy(), y_ref, c, TOL_FP32, "route on input")
    assert m.status() == 0
    m.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("E,d_model,d_ff,T,top_k", [
    (4, 512, 256, 3, 2),
    (16, 1024, 512, 8, 1),
])
def test_moe_ffn_route_on_input(monkeypatch, fmt, fused, E, d_model, d_ff, T, top_k):
    """The Llama 4 expert FFN: r scales the expert input, the slots are summed
    without it; checked against the oracle's input form, and shown to differ
    from the output form by more than the bound."""
    if not fused:
        monkeypatch.setenv("QMM_MOE_NOFUSE", "1")
    wg, wu, wd, ids, r, X = _ffn_case(E, d_model, d_ff, T, top_k, seed=40 + E, fmt=fmt)
    r = (r * np.float32(4.0)).astype(np.float32)  # far from 1, so the forms separate
    y_ref, c = _ffn_bound_input(wg, wu, wd, E, d_model, d_ff, ids, r, X, fmt)
    hs = [q.Matrix(fmt, E * d_ff, d_model, to_dev(wg)),
          q.Matrix(fmt, E * d_ff, d_model, to_dev(wu)),
          q.Matrix(fmt, E * d_model, d_ff, to_dev(wd))]
    Y = torch.full((T, d_model), float("nan"), dtype=torch.float32, device="cuda")
    q.moe_ffn(hs[0].h, hs[1].h, hs[2].h, E, to_dev(ids), T, top_k, to_dev(X), to_dev(r), Y,
              route_on_input=True)
    torch.cuda.synchronize()
    y = Y.cpu().numpy()
    assert_close_to_oracle(y, y_ref, c, TOL_FP32, "ffn route on input")
    y_out = oracle.moe_ffn(fmt, wg, wu, wd, E, d_model, d_ff, ids, X, r, nthreads=NTHREADS)
    assert np.max(np.abs(y_out - y_ref) - 1e-4 * c) > 0  # the other order is outside the bound
    assert hs[0].status() == 0
    for h in hs:
        h.close()


def test_moe_route_on_input_refusals():
    E, Ne, K = 4, 32, 256
    w, m = _stacked(E, Ne, K, seed=5)
    ids, r = _ids_uniform(2, E, 2, seed=6)
    X = synth.activations(2, K, seed=7)
    Y = torch.zeros((4, Ne), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.moe_gemv(m.h, E, to_dev(ids), 2, 2, to_dev(X), False, None, Y, route_on_input=True)
    assert ei.value.status == q.ERR_NULL
    ids_d, X_d, r_d = to_dev(ids), to_dev(X), to_dev(r)
    rc = q.lib().qmm_moe_gemv(ctypes.c_void_p(m.h), E, ctypes.c_void_p(ids_d.data_ptr()), 2, 2,
                              ctypes.c_void_p(X_d.data_ptr()), 0, ctypes.c_void_p(r_d.data_ptr()),
                              2, ctypes.c_void_p(Y.data_ptr()), None)
    assert rc == q.ERR_SHAPE and "route_on_input" in q.last_error()
    m.close()
