"""The oracle's pins catch plausible mistakes (no GPU).

Each case rebuilds the oracle from a copy of its C source with one mistake
planted (a swapped nibble, a wrong sign, a wrong index, a dropped term, a
wrong rounding...), points the oracle module at that build, and runs the
pins of tests/test_oracle.py and tests/test_oracle_formats.py against it:
at least one pin must fail.  A
control build of the unchanged source must pass every pin, so a failure
means the planted mistake was seen.  The planted mistake lives only in the
temporary copy; the real oracle is untouched and is restored afterwards."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle as pins
from tests import test_oracle_formats as format_pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "qmm_oracle.c")

# (name, [(text in qmm_oracle.c, replacement), ...])
MUTANTS = [
    ("nibble halves swapped", [("return qs[32 * c + l] & 15;", "return qs[32 * c + l] >> 4;"),
                               ("return qs[32 * c + l - 32] >> 4;", "return qs[32 * c + l - 32] & 15;")]),
    ("min term added", [("w[i] = d * sc * q - dmin * m;", "w[i] = d * sc * q + dmin * m;")]),
    ("min term dropped", [("w[i] = d * sc * q - dmin * m;", "w[i] = d * sc * q;")]),
    ("scale and min swapped", [("*sc = sc12[j] & 63;\n        *m = sc12[j + 4] & 63;",
                                "*m = sc12[j] & 63;\n        *sc = sc12[j + 4] & 63;")]),
    ("packing shift wrong", [("((sc12[j - 4] >> 6) << 4)", "((sc12[j - 4] >> 6) << 2)")]),
    ("packing byte off by one", [("*sc = (sc12[j + 4] & 15)", "*sc = (sc12[j + 3] & 15)")]),
    ("sub-block index wrong", [("*sub = 2 * c + 1;", "*sub = 2 * c;")]),
    ("fp16 exponent bias", [("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)")]),
    ("fp16 subnormal scale", [("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);")]),
    ("q8_0 read unsigned", [("        if (q > 127)\n            q -= 256; /* two's complement int8 */\n", "")]),
    ("gemv skips the last weight", [("for (int64_t k = 0; k < K; ++k) {\n                        double p",
                                     "for (int64_t k = 0; k < K - 1; ++k) {\n                        double p")]),
    ("gemv reads x reversed", [("double p = wr[k] * (double)x[k];",
                                "double p = wr[k] * (double)x[K - 1 - k];")]),
    ("bf16 truncates", [("if (rest > 0x8000u || (rest == 0x8000u && (lower & 1u)))", "if (0)")]),
    ("bf16 ties away", [("(rest == 0x8000u && (lower & 1u))", "(rest == 0x8000u)")]),
    ("prefill uses exact weights", [("s += wb[k] * xv;", "s += wr[k] * xv;")]),
    ("silu sign", [("h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "h[i] = g[i] / (1.0 + exp(g[i])) * u[i];")]),
    ("q5_k fifth bit from the wrong sub-block", [("(2 * c + (l >= 32))", "(2 * c)")]),
    ("q5_k fifth bit weight", [("int q5 = lo | (hi << 4);", "int q5 = lo | (hi << 3);")]),
    ("q5_k min term dropped", [("w[i] = d * sc * q5 - dmin * m;", "w[i] = d * sc * q5;")]),
    ("q5_k fifth bit byte", [("(qh[l % 32] >>", "(qh[l / 2] >>")]),
    ("q6_k offset", [("int q = (lo | (hi << 4)) - 32;", "int q = (lo | (hi << 4)) - 31;")]),
    ("q6_k scale group of 32", [("scales[i / 16]", "scales[i / 32]")]),
    ("q6_k scale read unsigned", [("        if (sc > 127)\n            sc -= 256; /* int8 scale */\n", "")]),
    ("q6_k high-bit shift", [("(qh[32 * n + l] >> (2 * t)) & 3", "(qh[32 * n + l] >> t) & 3")]),
    ("q6_k low-bit byte", [("ql[64 * n + 32 * (t & 1) + l]", "ql[64 * n + 32 * (t >> 1) + l]")]),
    ("q6_k nibble choice", [("(t >= 2) ? (byte >> 4) : (byte & 15)", "(t & 1) ? (byte >> 4) : (byte & 15)")]),
    ("q6_k d from the front", [("blk[208] | (blk[209] << 8)", "blk[0] | (blk[1] << 8)")]),
    ("iq4_nl nibble halves swapped", [("w[j] = d * iq4nl_table[qs[j] & 15];", "w[j] = d * iq4nl_table[qs[j] >> 4];"),
                                      ("w[16 + j] = d * iq4nl_table[qs[j] >> 4];", "w[16 + j] = d * iq4nl_table[qs[j] & 15];")]),
    ("iq4_nl interleaved order", [("w[16 + j] = d * iq4nl_table[qs[j] >> 4];", "w[16 + j] = d * iq4nl_table[qs[15 - j] >> 4];")]),
]


def _pin_calls():
    """Every pin of the two oracle pin modules with its parameter sets."""
    calls = []
    for mod in (pins, format_pins):
        for name in dir(mod):
            if not name.startswith("test_"):
                continue
            fn = getattr(mod, name)
            marks = getattr(fn, "pytestmark", [])
            params = [m for m in marks if m.name == "parametrize"]
            label = f"{mod.__name__.rsplit('.', 1)[-1]}::{name}"
            if not params:
                calls.append((label, fn, {}))
                continue
            argname, values = params[0].args[0], params[0].args[1]
            for v in values:
                calls.append((f"{label}[{v}]", fn, {argname: v}))
    return calls


def _failing_pins(tmp_path, monkeypatch, src):
    """Build `src` as the oracle and return the pins that fail against it."""
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src)
    mlib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                    "-shared", "-fPIC", str(msrc), "-o", str(mlib), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_SRC", str(msrc))
    monkeypatch.setattr(oracle, "_LIB", str(mlib))
    monkeypatch.setattr(oracle, "_lib", None)
    failed = []
    for pname, fn, kw in _pin_calls():
        try:
            fn(**kw)
        except Exception:  # an assertion (or a refusal) in the pin
            failed.append(pname)
    monkeypatch.setattr(oracle, "_lib", None)  # drop the copied library before the real one returns
    return failed


needs_gcc = pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc is needed to build copies")


@needs_gcc
def test_unchanged_copy_passes_every_pin(tmp_path, monkeypatch):
    assert _failing_pins(tmp_path, monkeypatch, open(SRC).read()) == []


@needs_gcc
@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor for '{name}' not found once: {old!r}"
        src = src.replace(old, new)
    assert _failing_pins(tmp_path, monkeypatch, src), f"no pin caught the planted mistake '{name}'"
