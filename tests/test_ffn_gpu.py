"""GPU parity of the dense SwiGLU FFN for one token (qmm_ffn_decode) against
an oracle composition: h = silu(Wg x) * (Wu x), y = Wd h.

Bounds carry the GEMV bound (1e-4 of sum|w x|) through SwiGLU to first order
(|silu'| <= 1.1) plus the rounding of h itself, and through the down
projection as sum|Wd| a with a the bound's weights on h."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests._util import TOL_FP32, assert_close_to_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("quantized_gguf_dequant_gb300")

NT = max(1, oracle.max_threads())


def _case(fmt, d_model, d_ff, seed):
    wg = synth.matrix(fmt, d_ff, d_model, seed)
    wu = synth.matrix(fmt, d_ff, d_model, seed + 1)
    wd = synth.matrix(fmt, d_model, d_ff, seed + 2)
    x = synth.activations(1, d_model, seed + 3)[0]
    return wg, wu, wd, x


def _reference(fmt, wg, wu, wd, x, d_model, d_ff):
    """(h_ref, bound on h, y_ref, bound on y), all from the oracle."""
    g, cg = oracle.gemv(fmt, wg, d_ff, d_model, x[None], nthreads=NT)
    u, cu = oracle.gemv(fmt, wu, d_ff, d_model, x[None], nthreads=NT)
    h = oracle.swiglu(g[0], u[0])
    sg = oracle.swiglu(g[0], np.ones_like(g[0]))  # silu(g)
    a = np.abs(h) + 1.1 * np.abs(u[0]) * cg[0] + np.abs(sg) * cu[0]
    y, _ = oracle.gemv(fmt, wd, d_model, d_ff, h.astype(np.float32)[None], nthreads=NT)
    _, cd = oracle.gemv(fmt, wd, d_model, d_ff, a.astype(np.float32)[None], nthreads=NT)
    return h, a * 1.0001, y[0], cd[0] * 1.0001


def _run(hs, x, d_model, d_ff, stream=None):
    h = torch.full((d_ff,), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((d_model,), float("nan"), dtype=torch.float32, device="cuda")
    q.ffn_decode(hs[0].h, hs[1].h, hs[2].h, to_dev(x), h, y, stream)
    torch.cuda.synchronize()
    return h.cpu().numpy(), y.cpu().numpy()


def _handles(fmt, wg, wu, wd, d_model, d_ff):
    return [q.Matrix(fmt, d_ff, d_model, to_dev(wg)), q.Matrix(fmt, d_ff, d_model, to_dev(wu)),
            q.Matrix(fmt, d_model, d_ff, to_dev(wd))]


@pytest.mark.parametrize("fused", ["decode", "tc", "no"])
@pytest.mark.parametrize("fmt,d_model,d_ff", [
    (q.Q4_K, 256, 256),
    (q.Q4_K, 512, 768),
    (q.Q4_K, 1024, 2816),     # more (gate, up) tile pairs than CTAs
    (q.Q4_K, 2048, 5632),
    (q.Q4_K, 4096, 14336),    # Llama-3.1-8B
    (q.Q4_K, 40960, 256),     # long activations: K sliced (decode kernel) / grouped route
    (q.Q8_0, 512, 768),
    (q.Q8_0, 4096, 14336),
    (q.Q5_K, 2048, 5632),
    (q.Q6_K, 2048, 6144),
    (q.IQ4_NL, 1024, 2816),
])
def test_ffn_decode(monkeypatch, fused, fmt, d_model, d_ff):
    """SwiGLU fused into the decode kernel's output phase ('decode': gate and
    up tiles interleaved in one launch), into the earlier tensor-core
    kernel's pair mode ('tc', Q4_K), or as its own kernel ('no')."""
    if fused == "no":
        monkeypatch.setenv("QMM_FFN_NOFUSE", "1")
    elif fused == "tc":
        monkeypatch.setenv("QMM_FFN_PATH", "tc")
    wg, wu, wd, x = _case(fmt, d_model, d_ff, seed=d_model + d_ff + fmt)
    h_ref, ch, y_ref, cy = _reference(fmt, wg, wu, wd, x, d_model, d_ff)
    hs = _handles(fmt, wg, wu, wd, d_model, d_ff)
    h, y = _run(hs, x, d_model, d_ff)
    what = f"fmt={fmt} d_model={d_model} d_ff={d_ff} fused={fused}"
    assert_close_to_oracle(h, h_ref, ch, TOL_FP32, "h " + what)
    assert_close_to_oracle(y, y_ref, cy, TOL_FP32, "y " + what)
    for m in hs:
        assert m.status() == 0
        m.close()


@pytest.mark.parametrize("fused,launches", [(True, 2), (False, 3)])
def test_ffn_decode_launches(monkeypatch, fused, launches):
    """Fused: one gate/up/SwiGLU launch and the down GEMV.  Unfused: the
    grouped gate/up GEMV, SwiGLU and the down GEMV."""
    if not fused:
        monkeypatch.setenv("QMM_FFN_NOFUSE", "1")
    d_model, d_ff = 1024, 2816
    wg, wu, wd, x = _case(q.Q4_K, d_model, d_ff, seed=5)
    hs = _handles(q.Q4_K, wg, wu, wd, d_model, d_ff)
    _run(hs, x, d_model, d_ff)  # first call may set up scratch
    n0 = q.launch_count()
    _run(hs, x, d_model, d_ff)
    assert q.launch_count() - n0 == launches
    for m in hs:
        m.close()


def test_ffn_decode_graph_replay():
    """Captured after one eager call, chained layers replay to the eager bits."""
    d_model, d_ff, L = 1024, 2816, 4
    wg, wu, wd, x = _case(q.Q4_K, d_model, d_ff, seed=9)
    hs = _handles(q.Q4_K, wg, wu, wd, d_model, d_ff)
    xs = [to_dev(x)] + [torch.zeros(d_model, dtype=torch.float32, device="cuda") for _ in range(L)]
    hb = torch.zeros(d_ff, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def chain():
        for i in range(L):
            q.ffn_decode(hs[0].h, hs[1].h, hs[2].h, xs[i], hb, xs[i + 1], s)

    with torch.cuda.stream(s):
        chain()
    s.synchronize()
    eager = xs[L].clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for t in xs[1:]:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(xs[L].view(torch.int32), eager.view(torch.int32))
    # the first layer's output against the oracle composition
    xs1 = xs[1].cpu().numpy()
    _, _, y_ref, cy = _reference(q.Q4_K, wg, wu, wd, x, d_model, d_ff)
    assert_close_to_oracle(xs1, y_ref, cy, TOL_FP32, "graph layer 0")
    for m in hs:
        m.close()


def test_ffn_decode_refusals():
    d_model, d_ff = 512, 768
    wg, wu, wd, x = _case(q.Q4_K, d_model, d_ff, seed=3)
    hg, hu, hd = _handles(q.Q4_K, wg, wu, wd, d_model, d_ff)
    wrong = q.Matrix(q.Q4_K, d_ff, d_model, to_dev(wu))  # not d_model x d_ff
    h = torch.zeros(d_ff, dtype=torch.float32, device="cuda")
    y = torch.zeros(d_model, dtype=torch.float32, device="cuda")
    xd = to_dev(x)
    with pytest.raises(q.QmmError) as ei:
        q.ffn_decode(hg.h, hu.h, wrong.h, xd, h, y)
    assert ei.value.status == q.ERR_SHAPE
    with pytest.raises(q.QmmError) as ei:
        q.ffn_decode(hg.h, hd.h, hd.h, xd, h, y)  # up not the gate's shape
    assert ei.value.status == q.ERR_SHAPE
    hbig = torch.zeros(d_ff + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.ffn_decode(hg.h, hu.h, hd.h, xd, hbig[1:], y)  # h off 16-byte alignment
    assert ei.value.status == q.ERR_ALIGN
    for m in (hg, hu, hd, wrong):
        m.close()
