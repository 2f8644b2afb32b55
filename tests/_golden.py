"""Readers for the hand-written fixtures under tests/golden/ (no arithmetic
of the method here: the fixtures carry the expected values)."""
from __future__ import annotations

import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _expect(spec: str, n: int):
    out = {}
    for item in spec.split(","):
        where, val = item.split(":")
        v = float.fromhex(val) if val.startswith(("0x", "-0x")) else float(val)
        if "-" in where[1:]:
            a, b = where.split("-", 1)
            for i in range(int(a), int(b) + 1):
                out[i] = v
        else:
            out[int(where)] = v
    assert all(0 <= i < n for i in out)
    return out


def blocks():
    """Yield (fmt, name, block_bytes, {index: exact value})."""
    for line in _lines("blocks.txt"):
        parts = line.split()
        fmt, name = parts[0], parts[1]
        kv = dict(p.split("=", 1) for p in parts[2:])
        d = bytes.fromhex(kv["d"])[::-1]  # fixtures give the fp16 as a number
        if fmt == "q4k":
            dmin = bytes.fromhex(kv["dmin"])[::-1]
            sc12 = bytes.fromhex(kv["sc12"])
            assert len(sc12) == 12
            qs = bytearray(128)
            spec = kv["q"]
            if spec.startswith("all:"):
                qs = bytearray([int(spec[4:], 16)] * 128)
            else:
                for item in spec.split(","):
                    i, v = item.split(":")
                    qs[int(i)] = int(v, 16)
            blk = d + dmin + sc12 + bytes(qs)
            assert len(blk) == 144
            yield 12, name, blk, _expect(kv["expect"], 256)
        elif fmt == "q8_0":
            q = [int(v) for v in kv["q"].split(",")]
            assert len(q) == 32
            blk = d + bytes([(v + 256) % 256 for v in q])
            assert len(blk) == 34
            yield 8, name, blk, _expect(kv["expect"], 32)
        else:
            raise ValueError(fmt)


def scale_min_table():
    """Yield (sc12 bytes, [sc0..sc7], [m0..m7])."""
    for line in _lines("q4k_scale_min.txt"):
        parts = line.split()
        sc12 = bytes.fromhex(parts[0])
        vals = [int(v) for v in parts[1:]]
        assert len(sc12) == 12 and len(vals) == 16
        yield sc12, vals[:8], vals[8:]
