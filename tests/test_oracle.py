"""Pins for the CPU oracle (no GPU).

The oracle is trusted only after it is tied to things other than itself:
hand-worked blocks (tests/golden/), library routines that decode the same
encodings (numpy/struct binary16, torch bfloat16), an independent bit-level
evaluator written here from the format text, closed forms (one-hot inputs,
linearity, all-zero quants), and reductions of the expert layer to the dense
case.  Each check is built so that a plausible slip in the oracle (a swapped
nibble, a wrong packing shift, a dropped min term, a transposed operand)
fails at least one of them.
"""
from __future__ import annotations

import math
import struct

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth
from tests import _golden

Q4_K, Q8_0 = oracle.Q4_K, oracle.Q8_0


# ------------------------------------------------------------------ binary16

def test_half_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_float64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, oracle.half_to_float64(0x8000)) == -1.0


# ------------------------------------------------------------------ Q4_K scales

def test_scale_min_hand_table():
    for sc12, scs, ms in _golden.scale_min_table():
        for j in range(8):
            assert oracle.q4k_scale_min(sc12, j) == (scs[j], ms[j]), (sc12.hex(), j)


def _pack_scale_min(sc, m):
    """Independent packer: place each 6-bit field at the bit positions the
    packing assigns it, viewing the 12 bytes as one little-endian integer."""
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    S = 0
    for j in range(4):
        S |= sc[j] << (8 * j)
        S |= m[j] << (8 * (j + 4))
    for j in range(4, 8):
        S |= (sc[j] & 15) << (8 * (j + 4))
        S |= (sc[j] >> 4) << (8 * (j - 4) + 6)
        S |= (m[j] & 15) << (8 * (j + 4) + 4)
        S |= (m[j] >> 4) << (8 * j + 6)
    return S.to_bytes(12, "little")


def test_scale_min_round_trip_all_values():
    rng = np.random.default_rng(7)
    # every (sc, m) pair in every slot, with random other fields
    for j in range(8):
        for v in range(64):
            sc = list(rng.integers(0, 64, 8))
            m = list(rng.integers(0, 64, 8))
            sc[j] = v
            m[j] = 63 - v
            b = _pack_scale_min(sc, m)
            for jj in range(8):
                assert oracle.q4k_scale_min(b, jj) == (sc[jj], m[jj])


def test_packing_is_a_bijection():
    # the packer must use each of the 96 bits exactly once
    used = 0
    for j in range(8):
        for field in ("sc", "m"):
            for bit in range(6):
                sc = [0] * 8
                m = [0] * 8
                (sc if field == "sc" else m)[j] = 1 << bit
                S = int.from_bytes(_pack_scale_min(sc, m), "little")
                assert bin(S).count("1") == 1
                assert used & S == 0
                used |= S
    assert used == (1 << 96) - 1


# ------------------------------------------------------------------ blocks

def test_golden_blocks():
    n = 0
    for fmt, name, blk, expect in _golden.blocks():
        w = oracle.dequant_block(fmt, blk)
        for i, v in expect.items():
            assert w[i] == v, (name, i, w[i], v)
        n += 1
    assert n >= 9


def _naive_q4k_block(blk: bytes):
    """Bit-level evaluator written from the format text, independent of the
    C oracle: the fp16 fields via struct, the 6-bit fields and the nibbles
    read from the bytes viewed as little-endian integers."""
    d = struct.unpack("<e", blk[0:2])[0]
    dmin = struct.unpack("<e", blk[2:4])[0]
    S = int.from_bytes(blk[4:16], "little")
    Q = int.from_bytes(blk[16:144], "little")

    def bits(v, lo, n):
        return (v >> lo) & ((1 << n) - 1)

    out = []
    for i in range(256):
        c, l = divmod(i, 64)
        j = 2 * c + (1 if l >= 32 else 0)
        q = bits(Q, 8 * (32 * c + l % 32) + (4 if l >= 32 else 0), 4)
        if j < 4:
            sc = bits(S, 8 * j, 6)
            m = bits(S, 8 * (j + 4), 6)
        else:
            sc = bits(S, 8 * (j + 4), 4) | (bits(S, 8 * (j - 4) + 6, 2) << 4)
            m = bits(S, 8 * (j + 4) + 4, 4) | (bits(S, 8 * j + 6, 2) << 4)
        out.append(float(d) * sc * q - float(dmin) * m)
    return out


def _naive_q8_0_block(blk: bytes):
    d = struct.unpack("<e", blk[0:2])[0]
    return [float(d) * q for q in struct.unpack("<32b", blk[2:34])]


def test_random_blocks_vs_naive_evaluator():
    w4 = synth.q4k_matrix(8, 512, seed=11)
    for r in range(8):
        row = w4[r].tobytes()
        for b in range(2):
            blk = row[b * 144:(b + 1) * 144]
            assert list(oracle.dequant_block(Q4_K, blk)) == _naive_q4k_block(blk)
    w8 = synth.q8_0_matrix(4, 256, seed=12)
    for r in range(4):
        row = w8[r].tobytes()
        for b in range(8):
            blk = row[b * 34:(b + 1) * 34]
            assert list(oracle.dequant_block(Q8_0, blk)) == _naive_q8_0_block(blk)


def test_all_zero_quants_is_minus_dmin_m():
    rng = np.random.default_rng(3)
    for _ in range(50):
        blk = bytearray(rng.bytes(144))
        blk[16:] = bytes(128)
        d, dmin = struct.unpack("<ee", bytes(blk[0:4]))
        if not (math.isfinite(d) and math.isfinite(dmin)):
            continue
        w = oracle.dequant_block(Q4_K, bytes(blk))
        for j in range(8):
            _, m = oracle.q4k_scale_min(bytes(blk[4:16]), j)
            assert np.all(w[32 * j:32 * j + 32] == -float(dmin) * m)


def test_single_nibble_lands_on_its_weight():
    # d=1, dmin=0, all sc=1, m=0: w = q exactly
    base = bytearray(144)
    base[0:2] = b"\x00\x3c"
    base[4:16] = bytes.fromhex("010101010000000001010101")
    for byte in range(128):
        for hi in (0, 1):
            blk = bytearray(base)
            blk[16 + byte] = 0x70 if hi else 0x07
            w = oracle.dequant_block(Q4_K, bytes(blk))
            c, l = divmod(byte, 32)
            idx = 64 * c + l + 32 * hi
            expect = np.zeros(256)
            expect[idx] = 7.0
            assert np.array_equal(w, expect), (byte, hi)


def test_q8_0_d_one_gives_integers():
    blk = b"\x00\x3c" + bytes(range(256))[:32]
    w = oracle.dequant_block(Q8_0, blk)
    assert list(w) == list(range(32))
    blk = b"\x00\x3c" + bytes(range(224, 256))
    w = oracle.dequant_block(Q8_0, blk)
    assert list(w) == list(range(-32, 0))


def test_dequant_rows_matches_blocks():
    N, K = 5, 768
    w = synth.q4k_matrix(N, K, seed=5)
    full = oracle.dequant_rows(Q4_K, w, N, K)
    for r in range(N):
        for b in range(3):
            blk = w[r, b * 144:(b + 1) * 144].tobytes()
            assert np.array_equal(full[r, b * 256:(b + 1) * 256],
                                  oracle.dequant_block(Q4_K, blk))
    part = oracle.dequant_rows(Q4_K, w, N, K, row0=2, nrows=2)
    assert np.array_equal(part, full[2:4])


# ------------------------------------------------------------------ GEMV

@pytest.mark.parametrize("fmt", [Q4_K, Q8_0])
def test_gemv_one_hot_extracts_columns(fmt):
    N, K = 6, 512
    w = synth.matrix(fmt, N, K, seed=21)
    W = oracle.dequant_rows(fmt, w, N, K)
    for k in (0, 1, 31, 32, 63, 64, 255, 256, 300, 511):
        x = np.zeros(K, np.float32)
        x[k] = 1.0
        y, c = oracle.gemv(fmt, w, N, K, x)
        assert np.array_equal(y, W[:, k])
        assert np.array_equal(c, np.abs(W[:, k]))


@pytest.mark.parametrize("fmt", [Q4_K, Q8_0])
def test_gemv_brute_force_vs_naive(fmt):
    for N, K in ((1, 256), (3, 256), (4, 512)):
        w = synth.matrix(fmt, N, K, seed=N * 1000 + K)
        x = synth.activations(1, K, seed=K)[0]
        y, c = oracle.gemv(fmt, w, N, K, x)
        nb = K // (256 if fmt == Q4_K else 32)
        bb = 144 if fmt == Q4_K else 34
        dec = _naive_q4k_block if fmt == Q4_K else _naive_q8_0_block
        for r in range(N):
            row = w[r].tobytes()
            wr = []
            for b in range(nb):
                wr += dec(row[b * bb:(b + 1) * bb])
            prods = [wv * float(xv) for wv, xv in zip(wr, x)]
            assert math.isclose(y[r], math.fsum(prods), rel_tol=0, abs_tol=1e-12 * sum(map(abs, prods)))
            assert math.isclose(c[r], math.fsum(map(abs, prods)), rel_tol=1e-14)


def test_gemv_linearity_and_batch():
    N, K = 7, 1024
    w = synth.q4k_matrix(N, K, seed=31)
    X = synth.activations(3, K, seed=32)
    Y, C = oracle.gemv(Q4_K, w, N, K, X)
    for m in range(3):
        y, c = oracle.gemv(Q4_K, w, N, K, X[m])
        assert np.array_equal(Y[m], y) and np.array_equal(C[m], c)
    a, b = 0.75, -2.0
    xs = (a * X[0].astype(np.float64) + b * X[1].astype(np.float64)).astype(np.float32)
    ys, _ = oracle.gemv(Q4_K, w, N, K, xs)
    # xs was rounded to fp32, so compare against the exact product of the rounded input
    W = oracle.dequant_rows(Q4_K, w, N, K)
    assert np.allclose(ys, W @ xs.astype(np.float64), rtol=0, atol=1e-12 * np.abs(W) @ np.abs(xs))
    assert np.allclose(a * Y[0] + b * Y[1], W @ (a * X[0].astype(np.float64) + b * X[1]),
                       rtol=0, atol=1e-11 * (np.abs(W) @ np.abs(X[0]) + np.abs(W) @ np.abs(X[1])))


def test_gemv_rows_subset_and_threads():
    N, K = 64, 512
    w = synth.q8_0_matrix(N, K, seed=41)
    x = synth.activations(2, K, seed=42)
    Y, C = oracle.gemv(Q8_0, w, N, K, x, nthreads=1)
    Y4, C4 = oracle.gemv(Q8_0, w, N, K, x, nthreads=4)
    assert np.array_equal(Y, Y4) and np.array_equal(C, C4)
    rows = [63, 0, 17, 17]
    Ys, Cs = oracle.gemv(Q8_0, w, N, K, x, rows=rows)
    assert np.array_equal(Ys, Y[:, rows]) and np.array_equal(Cs, C[:, rows])


def test_gemv_zero_x_is_exactly_zero():
    N, K = 3, 256
    w = synth.q4k_matrix(N, K, seed=1)
    y, c = oracle.gemv(Q4_K, w, N, K, np.zeros(K, np.float32))
    assert np.all(y == 0) and np.all(c == 0)


def test_bad_arguments_are_rejected():
    w = synth.q4k_matrix(2, 256, seed=1)
    with pytest.raises(ValueError):
        oracle.row_bytes(Q4_K, 100)
    with pytest.raises(ValueError):
        oracle.gemv(Q4_K, w, 2, 256, np.zeros(256, np.float32), rows=[2])


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_vs_torch():
    import torch
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        # exact ties: low 16 bits 0x8000, both parities of the kept part
        (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32),
        (np.arange(1000, dtype=np.uint32) * 0x10000 + 0xBF808000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1e-45], np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_float(v) for v in vals], np.uint16)
    assert np.array_equal(got, ref)
    for b in (0x3F80, 0xC000, 0x0001, 0x7F7F):
        assert oracle.bf16_to_float64(b) == float(
            torch.from_numpy(np.array([b], np.uint16).view(np.int16)).view(torch.bfloat16).float().item())


def test_gemm_bf16_identity_and_rounding():
    import torch
    N, K = 5, 512
    w = synth.q4k_matrix(N, K, seed=51)
    W = oracle.dequant_rows(Q4_K, w, N, K)
    Wb = torch.from_numpy(W.astype(np.float32)).to(torch.bfloat16).double().numpy()
    # identity rows of X pick out the bf16 weights exactly
    ks = [0, 7, 255, 256, 511]
    X = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        X[i, k] = 0x3F80  # 1.0
    Y, C = oracle.gemm_bf16(w, N, K, X)
    for i, k in enumerate(ks):
        assert np.array_equal(Y[i], Wb[:, k])
        assert np.array_equal(C[i], np.abs(W[:, k]))
    Xr = synth.activations_bf16(2, K, seed=52)
    Y, _ = oracle.gemm_bf16(w, N, K, Xr)
    xd = torch.from_numpy(Xr.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(Y, xd @ Wb.T, rtol=1e-13, atol=1e-13)


def test_gemm_bf16_q8_0_identity_and_hand_values():
    """Q8_0 weights d*q are exact in fp32 (11 x 8 bits); the prefill takes
    them rounded to bf16: 0.1 (fp16 0x2e66) * 127 = 12.6968994140625 rounds
    to 12.6875 in bf16, 0.1 * -3 = -0.2999267578125 to -0.30078125."""
    import torch
    N, K = 3, 256
    rows = []
    for n in range(N):
        blocks = []
        for b in range(K // 32):
            q = np.zeros(32, np.int8)
            q[(5 * b + n) % 32] = 127
            q[(5 * b + n + 1) % 32] = -3
            blocks.append(struct.pack("<H", 0x2E66) + q.tobytes())
        rows.append(b"".join(blocks))
    w = np.frombuffer(b"".join(rows), np.uint8).copy()
    k0 = 5 * 0 + 0  # row 0, block 0: q[0] = 127, q[1] = -3
    X = np.zeros((2, K), np.uint16)
    X[0, k0] = 0x3F80
    X[1, k0 + 1] = 0x3F80
    Y, C = oracle.gemm_bf16(w, N, K, X, fmt=Q8_0)
    assert Y[0, 0] == 12.6875 and Y[1, 0] == -0.30078125
    assert C[0, 0] == 0.0999755859375 * 127
    W = oracle.dequant_rows(Q8_0, w, N, K)
    Wb = torch.from_numpy(W.astype(np.float32)).to(torch.bfloat16).double().numpy()
    Xr = synth.activations_bf16(3, K, seed=53)
    Y, _ = oracle.gemm_bf16(w, N, K, Xr, fmt=Q8_0)
    xd = torch.from_numpy(Xr.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(Y, xd @ Wb.T, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ SwiGLU / experts

def test_swiglu_closed_forms():
    from scipy.special import expit
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 2.5, -700.0, 700.0])
    u = np.array([5.0, 2.0, 2.0, 1.0, 1.0, -3.0, 1.0, 1.0])
    h = oracle.swiglu(g, u)
    assert h[0] == 0.0
    assert np.allclose(h, g * expit(g) * u, rtol=1e-15, atol=0)
    assert math.isclose(h[3], 30.0, rel_tol=1e-12)
    assert abs(h[4]) < 1e-11


def _moe_fixture(seed=0, E=4, N_e=16, K=256, T=5, top_k=2, fmt=Q4_K):
    w = synth.matrix(fmt, E * N_e, K, seed=seed)
    ids, r = synth.router(T, E, top_k, seed=seed + 1)
    X = synth.activations(T, K, seed=seed + 2)
    return w, ids, r, X


def test_moe_top1_unit_weight_is_dense():
    E, N_e, K, T = 4, 16, 256, 6
    w, ids, r, X = _moe_fixture(E=E, N_e=N_e, K=K, T=T, top_k=1)
    Y, C = oracle.moe_gemv(Q4_K, w, E, N_e, K, ids, X, False, np.ones((T, 1)))
    for t in range(T):
        e = ids[t, 0]
        y, c = oracle.gemv(Q4_K, w, E * N_e, K, X[t], rows=np.arange(e * N_e, (e + 1) * N_e))
        assert np.array_equal(Y[t], y) and np.array_equal(C[t], c)


def test_moe_identical_experts_ignore_ids():
    E, N_e, K, T, top_k = 4, 16, 256, 5, 2
    one = synth.q4k_matrix(N_e, K, seed=9)
    w = np.concatenate([one] * E, axis=0)
    _, _, r, X = _moe_fixture(E=E, N_e=N_e, K=K, T=T, top_k=top_k)
    ids1 = np.array([[0, 1]] * T)
    ids2 = np.array([[3, 2]] * T)
    Y1, _ = oracle.moe_gemv(Q4_K, w, E, N_e, K, ids1, X, False, r)
    Y2, _ = oracle.moe_gemv(Q4_K, w, E, N_e, K, ids2, X, False, r)
    assert np.array_equal(Y1, Y2)
    y, _ = oracle.gemv(Q4_K, one, N_e, K, X)
    assert np.allclose(Y1, r.astype(np.float64).sum(axis=1, keepdims=True) * y, rtol=1e-13, atol=0)


def test_moe_combined_equals_weighted_slots():
    E, N_e, K, T, top_k = 8, 8, 512, 4, 3
    w, ids, r, X = _moe_fixture(E=E, N_e=N_e, K=K, T=T, top_k=top_k, fmt=Q8_0)
    S, SC = oracle.moe_gemv(Q8_0, w, E, N_e, K, ids, X, False)
    Y, C = oracle.moe_gemv(Q8_0, w, E, N_e, K, ids, X, False, r)
    ref = np.einsum("ts,tsn->tn", r.astype(np.float64), S.reshape(T, top_k, N_e))
    assert np.allclose(Y, ref, rtol=1e-14, atol=0)
    # per-slot inputs: X[t*top_k+s] replicated from X[t] gives the same result
    Xs = np.repeat(X, top_k, axis=0)
    S2, _ = oracle.moe_gemv(Q8_0, w, E, N_e, K, ids, Xs, True)
    assert np.array_equal(S, S2)


def test_moe_ffn_matches_composition():
    E, D, F, T, top_k = 4, 256, 256, 3, 2
    wg = synth.q4k_matrix(E * F, D, seed=61)
    wu = synth.q4k_matrix(E * F, D, seed=62)
    wd = synth.q4k_matrix(E * D, F, seed=63)
    ids, r = synth.router(T, E, top_k, seed=64)
    X = synth.activations(T, D, seed=65)
    y = oracle.moe_ffn(Q4_K, wg, wu, wd, E, D, F, ids, X, r)
    Wg = oracle.dequant_rows(Q4_K, wg, E * F, D)
    Wu = oracle.dequant_rows(Q4_K, wu, E * F, D)
    Wd = oracle.dequant_rows(Q4_K, wd, E * D, F)
    ref = np.zeros((T, D))
    for t in range(T):
        for s in range(top_k):
            e = ids[t, s]
            g = Wg[e * F:(e + 1) * F] @ X[t].astype(np.float64)
            u = Wu[e * F:(e + 1) * F] @ X[t].astype(np.float64)
            h = g / (1 + np.exp(-g)) * u
            ref[t] += r[t, s] * (Wd[e * D:(e + 1) * D] @ h)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


# ------------------------------------------------------------------ generator

def test_generator_fields():
    w = synth.q4k_matrix(64, 1024, seed=3)
    blocks = w.reshape(-1, 144)
    d = blocks[:, 0:2].copy().view("<f2").astype(np.float64)
    dmin = blocks[:, 2:4].copy().view("<f2").astype(np.float64)
    assert d.min() >= 9.99e-5 and d.max() <= 1.0001e-3
    assert dmin.min() >= 9.99e-5 and dmin.max() <= 1.0001e-3
    q8 = synth.q8_0_matrix(64, 1024, seed=3).reshape(-1, 34)
    q = q8[:, 2:].view(np.int8)
    assert q.min() == -127 and q.max() == 127
    ids, r = synth.router(32, 64, 8, seed=1)
    assert all(len(set(row)) == 8 for row in ids)
    assert np.all(np.diff(r, axis=1) <= 0)
    assert np.array_equal(synth.q4k_matrix(3, 256, 5), synth.q4k_matrix(3, 256, 5))


# ------------------------------------------------------------- routing on input

def _q8_0_diagonal(n: int, q_of_row) -> np.ndarray:
    """n x n Q8_0 matrix (one 32-weight block per row when n = 32), d = 1,
    weight (i, i) = q_of_row(i) and 0 elsewhere: its exact value is the
    diagonal matrix diag(q_of_row(i))."""
    assert n == 32
    rows = []
    for i in range(n):
        q = np.zeros(32, np.int8)
        q[i] = q_of_row(i)
        rows.append(struct.pack("<e", 1.0) + q.tobytes())
    return np.frombuffer(b"".join(rows), np.uint8).copy()


def test_moe_ffn_route_on_input_closed_form():
    """Llama 4 applies the routing weight to the expert's input ("Frink
    Inference: the Rust alternative to llama.cpp", "Architecture coverage:
    100 models with evidence").  With diagonal experts every output is a
    scalar closed form: expert 0 has Wg = I, Wu = 2I, Wd = I; expert 1 has
    Wg = 3I, Wu = I, Wd = -I.  Input form:  y = sum_s Wd (silu(r Wg x) * (r Wu x));
    output form: y = sum_s r Wd (silu(Wg x) * (Wu x))."""
    D = F = 32
    E = 2
    wg = np.concatenate([_q8_0_diagonal(32, lambda i: 1), _q8_0_diagonal(32, lambda i: 3)])
    wu = np.concatenate([_q8_0_diagonal(32, lambda i: 2), _q8_0_diagonal(32, lambda i: 1)])
    wd = np.concatenate([_q8_0_diagonal(32, lambda i: 1), _q8_0_diagonal(32, lambda i: -1)])
    ids = np.array([[0, 1], [1, 0], [0, 0]])
    r = np.array([[0.25, 1.5], [2.0, -0.5], [0.75, 0.125]], np.float32)
    X = np.linspace(-3.0, 3.0, 3 * D, dtype=np.float32).reshape(3, D)

    def silu(z):
        return z / (1.0 + math.exp(-z))

    gscale, uscale, dscale = {0: 1, 1: 3}, {0: 2, 1: 1}, {0: 1, 1: -1}
    ref_in = np.zeros((3, D))
    ref_out = np.zeros((3, D))
    for t in range(3):
        for s in range(2):
            e, rw = int(ids[t, s]), float(r[t, s])
            for i in range(D):
                x = float(X[t, i])
                ref_in[t, i] += dscale[e] * silu(gscale[e] * rw * x) * (uscale[e] * rw * x)
                ref_out[t, i] += rw * dscale[e] * silu(gscale[e] * x) * (uscale[e] * x)
    y_in = oracle.moe_ffn(Q8_0, wg, wu, wd, E, D, F, ids, X, r, route_on_input=True)
    y_out = oracle.moe_ffn(Q8_0, wg, wu, wd, E, D, F, ids, X, r)
    assert np.allclose(y_in, ref_in, rtol=1e-13, atol=1e-13)
    assert np.allclose(y_out, ref_out, rtol=1e-13, atol=1e-13)
    assert np.abs(y_in - y_out).max() > 0.1  # SwiGLU tells the two orders apart


def test_moe_route_on_input_unit_weights_and_linearity():
    """r = 1: the input form equals the output form exactly in the FFN; the
    expert GEMV is linear, so the scaled-input slot outputs equal r times the
    plain slot outputs to fp64 rounding."""
    E, D, F, T, top_k = 4, 256, 256, 3, 2
    wg = synth.q4k_matrix(E * F, D, seed=71)
    wu = synth.q4k_matrix(E * F, D, seed=72)
    wd = synth.q4k_matrix(E * D, F, seed=73)
    ids, r = synth.router(T, E, top_k, seed=74)
    X = synth.activations(T, D, seed=75)
    one = np.ones_like(r)
    y1 = oracle.moe_ffn(Q4_K, wg, wu, wd, E, D, F, ids, X, one, route_on_input=True)
    y2 = oracle.moe_ffn(Q4_K, wg, wu, wd, E, D, F, ids, X, one)
    assert np.allclose(y1, y2, rtol=1e-12, atol=1e-12 * np.abs(y2).max())
    S, _ = oracle.moe_gemv(Q4_K, wg, E, F, D, ids, X, False)
    Si, Ci = oracle.moe_gemv(Q4_K, wg, E, F, D, ids, X, False, r, route_on_input=True)
    ref = r.astype(np.float64).reshape(-1, 1) * S
    assert np.allclose(Si, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(Ci >= np.abs(Si) * (1 - 1e-12))
    with pytest.raises(ValueError):
        oracle.moe_gemv(Q4_K, wg, E, F, D, ids, X, False, None, route_on_input=True)


# ------------------------------------------------------------- Q8_K activations

def _q8k_fields(blk: bytes):
    d = struct.unpack("<f", blk[0:4])[0]
    q = list(struct.unpack("<256b", blk[4:260]))
    bsums = list(struct.unpack("<16h", blk[260:292]))
    return d, q, bsums


def test_q8_k_hand_block():
    """One block worked by hand: the largest |x| is -1.0 (index 5), so
    iscale = -127 / -1 = 127 exactly; 0.5 -> 63.5 -> 64 (half to even),
    -0.25 -> -31.75 -> -32, 0.75 -> 95.25 -> 95; d = 1/127 in binary32."""
    x = np.zeros(256, np.float32)
    x[5], x[6], x[7], x[20], x[255] = -1.0, 0.5, -0.25, 0.75, 1.0 / 127.0
    d, q, bs = _q8k_fields(oracle.quantize_q8_k(x).tobytes())
    assert d == float(np.float32(1.0) / np.float32(127.0))
    expect = {5: -127, 6: 64, 7: -32, 20: 95, 255: 1}
    for j in range(256):
        assert q[j] == expect.get(j, 0), j
    assert bs[0] == -127 + 64 - 32 and bs[1] == 95 and bs[15] == 1
    assert all(b == 0 for g, b in enumerate(bs) if g not in (0, 1, 15))


def test_q8_k_ties_to_even_and_first_max():
    # max = -63.5 -> iscale = 2 exactly: 0.25 -> 0.5 -> 0, 0.75 -> 1.5 -> 2,
    # 1.25 -> 2.5 -> 2, -1.25 -> -2.5 -> -2
    x = np.zeros(256, np.float32)
    x[0], x[1], x[2], x[3], x[4] = -63.5, 0.25, 0.75, 1.25, -1.25
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(x).tobytes())
    assert d == 0.5 and q[:5] == [-127, 0, 2, 2, -2]
    # equal |x| of both signs: the first one is the block's max
    y = np.zeros(256, np.float32)
    y[3], y[10] = -4.0, 4.0
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(y).tobytes())
    assert d > 0 and q[3] == -127 and q[10] == 127
    y[3], y[10] = 4.0, -4.0
    d, q, _ = _q8k_fields(oracle.quantize_q8_k(y).tobytes())
    assert d < 0 and q[3] == -127 and q[10] == 127


def test_q8_k_zero_block_and_bound():
    x = synth.activations(1, 1024, seed=81)[0].copy()
    x[256:512] = 0.0
    xq = oracle.quantize_q8_k(x)
    assert not xq[292:584].any()  # d = 0, q = 0, bsums = 0
    xh = oracle.dequant_q8_k(xq, 1024)
    for b in range(4):
        d, q, bs = _q8k_fields(xq[292 * b:292 * (b + 1)].tobytes())
        assert all(bs[g] == sum(q[16 * g:16 * g + 16]) for g in range(16))
        blk = x[256 * b:256 * (b + 1)].astype(np.float64)
        if d != 0.0:
            assert q[int(np.argmax(np.abs(blk)))] == -127
        assert np.all(np.abs(blk - xh[256 * b:256 * (b + 1)]) <= abs(d) * (0.5 + 2.0 ** -20))


def test_gemv_q8k_exact_when_x_is_on_the_grid():
    """x of integers in [-127, 127] with 127 the first largest element of
    every block: iscale = -1, q = -x, d = -1, so the dequantized activations
    are x itself and the integer-dot GEMV equals the f32 GEMV exactly."""
    K, N = 1024, 9
    rng = np.random.default_rng(82)
    x = rng.integers(-126, 127, K).astype(np.float32)
    x[0::256] = 127.0
    xq = oracle.quantize_q8_k(x)
    assert np.array_equal(oracle.dequant_q8_k(xq, K), x.astype(np.float64))
    w = synth.q4k_matrix(N, K, seed=83)
    y8, c8 = oracle.gemv_q8k(Q4_K, w, N, K, xq)
    y, c = oracle.gemv(Q4_K, w, N, K, x)
    assert np.array_equal(y8, y) and np.array_equal(c8, c)


def test_gemv_q8k_integer_regrouping_and_naive():
    """The llama.cpp grouping of the same sum -- per sub-block an integer dot
    of nibbles and codes scaled by sc, minus m times the block's code sums
    (bsums), then d_w * d_x -- computed here in Python integers from the raw
    bytes, equals the oracle; so does a naive loop over the naive block
    decoder."""
    K, N = 512, 3
    w = synth.q4k_matrix(N, K, seed=84)
    x = synth.activations(1, K, seed=85)[0]
    xq = oracle.quantize_q8_k(x)
    y8, c8 = oracle.gemv_q8k(Q4_K, w, N, K, xq)
    rb = K // 256 * 144
    wf = np.ascontiguousarray(w).reshape(-1)
    for n in range(N):
        tot = 0.0
        naive = 0.0
        for b in range(K // 256):
            blk = bytes(wf[n * rb + 144 * b:n * rb + 144 * (b + 1)])
            dx, qx, bs = _q8k_fields(xq[292 * b:292 * (b + 1)].tobytes())
            d = struct.unpack("<e", blk[0:2])[0]
            dmin = struct.unpack("<e", blk[2:4])[0]
            sumi = summ = 0
            for j in range(8):
                sc, m = oracle.q4k_scale_min(blk[4:16], j)
                c, hi = divmod(j, 2)
                dot = 0
                for l in range(32):
                    byte = blk[16 + 32 * c + l]
                    qw = (byte >> 4) if hi else (byte & 15)
                    dot += qw * qx[32 * j + l]
                sumi += sc * dot
                summ += m * (bs[2 * j] + bs[2 * j + 1])
            tot += float(d) * dx * sumi - float(dmin) * dx * summ
            wv = _naive_q4k_block(blk)
            naive += sum(wv[i] * dx * qx[i] for i in range(256))
        assert math.isclose(tot, y8[n], rel_tol=1e-12, abs_tol=1e-12 * c8[n])
        assert math.isclose(naive, y8[n], rel_tol=1e-12, abs_tol=1e-12 * c8[n])


def test_gemv_q8k_drift_within_stated_bound():
    """|y_q8k - y_f32| <= sum over blocks of (sum |w| over the block) * |d|/2:
    each activation moves by at most half a quantization step."""
    K, N = 2048, 16
    w = synth.q4k_matrix(N, K, seed=86)
    x = synth.activations(1, K, seed=87)[0]
    xq = oracle.quantize_q8_k(x)
    y8, _ = oracle.gemv_q8k(Q4_K, w, N, K, xq)
    y, _ = oracle.gemv(Q4_K, w, N, K, x)
    W = np.abs(oracle.dequant_rows(Q4_K, w, N, K)).reshape(N, K // 256, 256).sum(axis=2)
    dq = np.array([abs(struct.unpack("<f", xq[292 * b:292 * b + 4].tobytes())[0])
                   for b in range(K // 256)])
    bound = W @ (dq * (0.5 + 2.0 ** -20))
    assert np.all(np.abs(y8 - y) <= bound)
    assert np.any(np.abs(y8 - y) > 1e-3 * bound)  # the drift is real, not zero
