"""Pins for the oracle's further block formats: Q5_K, Q6_K and IQ4_NL (no GPU).

Each decoder is tied to a bit-level evaluator written here from the format
text (big integers over the block bytes, struct for the binary16 and int8
fields), to hand-built blocks whose values follow by inspection (one quant
set at a time, all-zero quants, distinct scales per group), and to the
closed forms of the GEMV (one-hot inputs).  The IQ4_NL code book itself is
part of the format; its values are pinned only through properties (16
integer entries of int8 range, strictly increasing, both signs): the entries
themselves are parity unpinned (no source here prints them), and conformance
to real GGUF files is unpinned, as for the other formats.
"""
from __future__ import annotations

import math
import struct

import numpy as np
import pytest

import oracle
from quantized_gguf_dequant_gb300 import synth

Q5_K, Q6_K, IQ4_NL = oracle.Q5_K, oracle.Q6_K, oracle.IQ4_NL
ONE = b"\x00\x3c"  # binary16 1.0


def _bits(v, lo, n):
    return (v >> lo) & ((1 << n) - 1)


# ------------------------------------------------------------------ evaluators

def _naive_q5k(blk: bytes):
    d, dmin = struct.unpack("<ee", blk[0:4])
    S = int.from_bytes(blk[4:16], "little")
    H = int.from_bytes(blk[16:48], "little")
    Q = int.from_bytes(blk[48:176], "little")
    out = []
    for i in range(256):
        c, l = divmod(i, 64)
        half = 1 if l >= 32 else 0
        j = 2 * c + half
        lo = _bits(Q, 8 * (32 * c + l % 32) + 4 * half, 4)
        hi = _bits(H, 8 * (l % 32) + j, 1)
        if j < 4:
            sc, m = _bits(S, 8 * j, 6), _bits(S, 8 * (j + 4), 6)
        else:
            sc = _bits(S, 8 * (j + 4), 4) | (_bits(S, 8 * (j - 4) + 6, 2) << 4)
            m = _bits(S, 8 * (j + 4) + 4, 4) | (_bits(S, 8 * j + 6, 2) << 4)
        out.append(float(d) * sc * (lo + 16 * hi) - float(dmin) * m)
    return out


def _naive_q6k(blk: bytes):
    L = int.from_bytes(blk[0:128], "little")
    H = int.from_bytes(blk[128:192], "little")
    scales = struct.unpack("<16b", blk[192:208])
    d = struct.unpack("<e", blk[208:210])[0]
    out = []
    for i in range(256):
        n, r = divmod(i, 128)
        t, l = divmod(r, 32)
        lo = _bits(L, 8 * (64 * n + 32 * (t % 2) + l) + 4 * (t // 2), 4)
        hi = _bits(H, 8 * (32 * n + l) + 2 * t, 2)
        out.append(float(d) * scales[i // 16] * (lo + 16 * hi - 32))
    return out


NAIVE = {Q5_K: _naive_q5k, Q6_K: _naive_q6k}


@pytest.mark.parametrize("fmt", [Q5_K, Q6_K])
def test_random_blocks_vs_naive_evaluator(fmt):
    nbytes, _ = oracle.BLOCK[fmt]
    w = synth.matrix(fmt, 6, 512, seed=fmt)
    for r in range(6):
        row = w[r].tobytes()
        for b in range(2):
            blk = row[b * nbytes:(b + 1) * nbytes]
            assert list(oracle.dequant_block(fmt, blk)) == NAIVE[fmt](blk), (r, b)


# ------------------------------------------------------------------ Q5_K

def _q5k_unit_block():
    """d = 1, dmin = 0, every scale 1, every min 0: w = q exactly."""
    blk = bytearray(176)
    blk[0:2] = ONE
    blk[4:16] = bytes.fromhex("010101010000000001010101")
    return blk


def test_q5k_low_bits_and_fifth_bit_land_on_their_weight():
    for l in range(32):
        for c in range(4):
            for half in (0, 1):
                blk = _q5k_unit_block()
                blk[48 + 32 * c + l] = 0x50 if half else 0x05
                blk[16 + l] = 1 << (2 * c + half)
                w = oracle.dequant_block(Q5_K, bytes(blk))
                expect = np.zeros(256)
                expect[64 * c + 32 * half + l] = 21.0  # 5 + 16
                assert np.array_equal(w, expect), (l, c, half)


def test_q5k_all_zero_quants_is_minus_dmin_m():
    rng = np.random.default_rng(4)
    for _ in range(30):
        blk = bytearray(rng.bytes(176))
        blk[16:] = bytes(160)
        d, dmin = struct.unpack("<ee", bytes(blk[0:4]))
        if not (math.isfinite(d) and math.isfinite(dmin)):
            continue
        w = oracle.dequant_block(Q5_K, bytes(blk))
        for j in range(8):
            _, m = oracle.q4k_scale_min(bytes(blk[4:16]), j)
            assert np.all(w[32 * j:32 * j + 32] == -float(dmin) * m)


def test_q5k_largest_quant_is_31():
    blk = _q5k_unit_block()
    blk[16:48] = b"\xff" * 32
    blk[48:176] = b"\xff" * 128
    assert np.all(oracle.dequant_block(Q5_K, bytes(blk)) == 31.0)


# ------------------------------------------------------------------ Q6_K

def _q6k_block(scales=(1,) * 16, d=ONE):
    blk = bytearray(210)
    blk[192:208] = struct.pack("<16b", *scales)
    blk[208:210] = d
    return blk


def test_q6k_zero_bytes_is_minus_32_d_scale():
    blk = _q6k_block(scales=tuple(range(-8, 8)))
    w = oracle.dequant_block(Q6_K, bytes(blk))
    assert np.array_equal(w, np.repeat(-32.0 * np.arange(-8, 8), 16))


def test_q6k_scale_per_group_of_16():
    # low bits 1, high bits 2 everywhere: q = 1 + 32 = 33, q - 32 = 1
    blk = _q6k_block(scales=tuple(range(1, 17)))
    blk[0:128] = b"\x11" * 128
    blk[128:192] = b"\xaa" * 64
    w = oracle.dequant_block(Q6_K, bytes(blk))
    assert np.array_equal(w, np.repeat(np.arange(1, 17, dtype=np.float64), 16))


def test_q6k_low_bits_land_on_their_weight():
    for byte in range(128):
        for nib in (0, 1):
            blk = _q6k_block()
            blk[byte] = 0x90 if nib else 0x09
            w = oracle.dequant_block(Q6_K, bytes(blk))
            n, rest = divmod(byte, 64)
            t = 2 * nib + rest // 32
            idx = 128 * n + 32 * t + rest % 32
            expect = np.full(256, -32.0)
            expect[idx] = 9.0 - 32.0
            assert np.array_equal(w, expect), (byte, nib)


def test_q6k_high_bits_land_on_their_weight():
    for byte in range(64):
        for t in range(4):
            blk = _q6k_block()
            blk[128 + byte] = 3 << (2 * t)
            w = oracle.dequant_block(Q6_K, bytes(blk))
            n, l = divmod(byte, 32)
            expect = np.full(256, -32.0)
            expect[128 * n + 32 * t + l] = 48.0 - 32.0
            assert np.array_equal(w, expect), (byte, t)


def test_q6k_negative_scale_and_d():
    blk = _q6k_block(scales=(-1,) * 16, d=b"\x00\xb8")  # d = -0.5
    blk[0:128] = b"\x33" * 128  # low bits 3, high bits 0: q - 32 = -29
    w = oracle.dequant_block(Q6_K, bytes(blk))
    assert np.all(w == -0.5 * -1 * -29)


# ------------------------------------------------------------------ IQ4_NL

def _iq4nl_table():
    """The code book as the oracle decodes it: code j sits in weight j of a
    block with d = 1 whose byte j holds code j in its low nibble."""
    blk = ONE + bytes(range(16))
    return oracle.dequant_block(IQ4_NL, blk)[:16]


def test_iq4nl_code_book_properties():
    T = _iq4nl_table()
    assert T.shape == (16,)
    assert np.all(np.diff(T) > 0)  # strictly increasing in the code
    assert np.all(T == np.round(T)) and np.all(np.abs(T) <= 127)  # int8 values
    assert T[0] < 0 < T[15]  # both signs
    # the same book for the high nibbles
    blk = ONE + bytes((j << 4) for j in range(16))
    w = oracle.dequant_block(IQ4_NL, blk)
    assert np.array_equal(w[16:], T) and np.all(w[:16] == T[0])


def test_iq4nl_nibble_order_and_scale():
    T = _iq4nl_table()
    rng = np.random.default_rng(9)
    for _ in range(20):
        qs = rng.integers(0, 256, 16).astype(np.uint8)
        d = float(np.float16(rng.uniform(-2, 2)))
        blk = struct.pack("<e", d) + qs.tobytes()
        w = oracle.dequant_block(IQ4_NL, blk)
        assert np.array_equal(w[:16], d * T[qs & 15])
        assert np.array_equal(w[16:], d * T[qs >> 4])


# ------------------------------------------------------------------ rows, GEMV

@pytest.mark.parametrize("fmt", [Q5_K, Q6_K, IQ4_NL])
def test_rows_are_blocks_in_order(fmt):
    nbytes, nw = oracle.BLOCK[fmt]
    N, K = 3, 768
    w = synth.matrix(fmt, N, K, seed=50 + fmt)
    assert w.shape == (N, oracle.row_bytes(fmt, K)) == (N, K // nw * nbytes)
    full = oracle.dequant_rows(fmt, w, N, K)
    for r in range(N):
        for b in range(K // nw):
            blk = w[r, b * nbytes:(b + 1) * nbytes].tobytes()
            assert np.array_equal(full[r, b * nw:(b + 1) * nw], oracle.dequant_block(fmt, blk))


@pytest.mark.parametrize("fmt", [Q5_K, Q6_K, IQ4_NL])
def test_gemv_one_hot_and_brute_force(fmt):
    N, K = 4, 512
    w = synth.matrix(fmt, N, K, seed=60 + fmt)
    W = oracle.dequant_rows(fmt, w, N, K)
    for k in (0, 15, 16, 31, 32, 255, 256, 511):
        x = np.zeros(K, np.float32)
        x[k] = 1.0
        y, c = oracle.gemv(fmt, w, N, K, x)
        assert np.array_equal(y, W[:, k]) and np.array_equal(c, np.abs(W[:, k]))
    x = synth.activations(1, K, seed=61)[0]
    y, c = oracle.gemv(fmt, w, N, K, x)
    for r in range(N):
        prods = [float(a) * float(b) for a, b in zip(W[r], x)]
        assert math.isclose(y[r], math.fsum(prods), rel_tol=0,
                            abs_tol=1e-12 * sum(map(abs, prods)))


def test_row_geometry_refusals():
    for fmt, bad in ((Q5_K, 128), (Q6_K, 300), (IQ4_NL, 48)):
        with pytest.raises(ValueError):
            oracle.row_bytes(fmt, bad)


def test_generator_fields():
    # d fields in [1e-4, 1e-3] (binary16), everything else uniform bytes
    w = synth.q6k_matrix(64, 256, seed=3)
    d = w[:, 208:210].copy().view("<f2").astype(np.float64)
    assert np.all((d >= 9.99e-5) & (d <= 1.0001e-3))
    w = synth.iq4nl_matrix(64, 256, seed=3).reshape(-1, 18)
    d = w[:, 0:2].copy().view("<f2").astype(np.float64)
    assert np.all((d >= 9.99e-5) & (d <= 1.0001e-3))
    w = synth.q5k_matrix(64, 256, seed=3)
    d = w[:, 0:4].copy().view("<f2").astype(np.float64)
    assert np.all((d >= 9.99e-5) & (d <= 1.0001e-3))
