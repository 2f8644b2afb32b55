"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every entry point include/qmm.h declares, and refuses bad arguments by name
on the host before touching the device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import quantized_gguf_dequant_gb300 as q
from quantized_gguf_dequant_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return q.lib()


def test_header_and_binding_agree():
    assert sorted(q.ENTRY_POINTS) == declared_entry_points()


def test_library_exports_every_entry_point(L):
    out = subprocess.run(["nm", "-D", "--defined-only", q.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (qmm_\w+)", out))
    missing = [f for f in declared_entry_points() if f not in exported]
    assert not missing, missing
    for f in declared_entry_points():
        assert hasattr(L, f)


def test_library_is_built_for_sm_103a_only():
    """Every translation unit and the link use one target: sm_103a."""
    from quantized_gguf_dequant_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    flags = build._flags()
    assert flags[:2] == build.ARCH
    assert not any("sm_" in f and "103a" not in f for f in flags)


def test_version(L):
    assert q.version() >= 100


def _create(fmt, N, K, ptr):
    h = ctypes.c_void_p()
    rc = q.lib().qmm_create(fmt, N, K, ctypes.c_void_p(ptr), ctypes.byref(h))
    return rc, q.last_error()


def test_create_refuses_by_name(L):
    rc, msg = _create(q.Q4_K, 16, 4096, 0)
    assert rc == q.ERR_NULL and "weight pointer" in msg
    rc, msg = _create(7, 16, 4096, 0x10000)
    assert rc == q.ERR_FORMAT and "format 7" in msg
    rc, msg = _create(q.Q4_K, 0, 4096, 0x10000)
    assert rc == q.ERR_SHAPE and "N = 0" in msg
    rc, msg = _create(q.Q4_K, 16, 1000, 0x10000)
    assert rc == q.ERR_SHAPE and "K = 1000" in msg and "256" in msg
    rc, msg = _create(q.Q8_0, 16, 100, 0x10000)  # Q8_0 rows take any multiple of 32
    assert rc == q.ERR_SHAPE and "K = 100" in msg and "32" in msg
    rc, msg = _create(q.Q4_K, 16, 4096, 0x10008)
    assert rc == q.ERR_ALIGN and "16-byte" in msg
    rc = q.lib().qmm_create(q.Q4_K, 16, 4096, ctypes.c_void_p(0x10000), None)
    assert rc == q.ERR_NULL


def test_format_ids_agree_with_the_header():
    text = open(HEADER).read()
    enum = re.search(r"typedef enum \{([^}]*)\} qmm_format;", text).group(1)
    ids = {k: int(v) for k, v in re.findall(r"QMM_(\w+)\s*=\s*(\d+)", enum)}
    assert ids == {"Q8_0": q.Q8_0, "Q4_K": q.Q4_K, "Q5_K": q.Q5_K, "Q6_K": q.Q6_K,
                   "IQ4_NL": q.IQ4_NL}
    # GGUF tensor-type ids
    assert (q.Q8_0, q.Q4_K, q.Q5_K, q.Q6_K, q.IQ4_NL) == (8, 12, 13, 14, 20)


def test_create_refuses_further_formats_by_name(L):
    for fmt in (q.Q5_K, q.Q6_K, q.IQ4_NL):
        rc, msg = _create(fmt, 16, 1000, 0x10000)
        assert rc == q.ERR_SHAPE and "K = 1000" in msg
        assert ("32" if fmt == q.IQ4_NL else "256") in msg
        rc, msg = _create(fmt, 16, 4096, 0x10008)
        assert rc == q.ERR_ALIGN and "16-byte" in msg
    rc, msg = _create(15, 16, 4096, 0x10000)
    assert rc == q.ERR_FORMAT and "format 15" in msg and "IQ4_NL = 20" in msg


def test_calls_on_null_handle_refuse(L):
    vp = ctypes.c_void_p
    assert L.qmm_gemv(None, vp(16), vp(16), None) == q.ERR_NULL
    assert "handle is NULL" in q.last_error()
    assert L.qmm_ffn_decode(None, None, None, vp(16), vp(16), vp(16), None) == q.ERR_NULL
    assert L.qmm_destroy(None) == q.ERR_NULL
    assert L.qmm_dequantize(None, 0, 1, vp(16), None) == q.ERR_NULL
    assert L.qmm_gemv_group(None, 1, vp(16), None, None) == q.ERR_NULL
    arr = (vp * 1)(vp(0))
    assert L.qmm_gemv_group(arr, 0, vp(16), arr, None) == q.ERR_SHAPE
    assert L.qmm_gemv_group(arr, 9, vp(16), arr, None) == q.ERR_SHAPE
