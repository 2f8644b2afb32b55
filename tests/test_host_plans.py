"""The library's launch planners on the host (no GPU): how the decode, batched,
prefill and fp32 GEMV launches cut their work, checked for every shape of a
grid against the invariants the kernels rely on (every weight covered once,
shared memory within the 227 KB a CTA may have, the grid within one CTA per
SM, scratch sized to what is written, in-kernel slice sums only where they
were measured to pay).

tests/host_plans.cu drives the planners through the library's own object
files; it makes no CUDA runtime call, so it runs here.
"""
from __future__ import annotations

import json
import os
import shutil
import subprocess

import pytest

from quantized_gguf_dequant_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152
SMEM_MAX = 227 * 1024

needs_nvcc = pytest.mark.skipif(not os.path.exists(qbuild.nvcc()) and shutil.which("nvcc") is None,
                                reason="nvcc is needed to link the planner driver")


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    qbuild.build()

    def objects():
        if not os.path.isdir(qbuild.BUILD):
            return []
        # the objects of the current sources only (a stale object of a
        # removed source would not link)
        names = {os.path.splitext(src)[0] + ".o" for src in qbuild.SOURCES}
        return sorted(os.path.join(qbuild.BUILD, f) for f in os.listdir(qbuild.BUILD)
                      if f in names)

    objs = objects()
    if len(objs) < len(qbuild.SOURCES):  # the library exists but its objects were removed
        qbuild.build(force=True)
        objs = objects()
    exe = str(tmp_path_factory.mktemp("plans") / "host_plans")
    subprocess.run([qbuild.nvcc(), "-std=c++17", "-O1", "-I" + os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "host_plans.cu"), *objs, "-o", exe, *qbuild.ARCH],
                   check=True, capture_output=True)
    env = {k: v for k, v in os.environ.items() if not k.startswith("QMM_")}  # defaults only
    out = subprocess.run([exe, str(SMS)], check=True, capture_output=True, text=True, env=env).stdout
    recs = [json.loads(line) for line in out.splitlines()]
    by = {}
    for r in recs:
        by.setdefault(r["kind"], []).append(r)
    return by


@needs_nvcc
def test_batched_plans(plans):
    rows = plans["tcb"]
    assert len(rows) == 8 * 6 * 16
    for p in rows:
        N, K, M = p["N"], p["K"], p["M"]
        NB, T = K // 256, (N + 15) // 16
        assert p["nt"] == (M + 3) // 4
        assert p["S"] >= 1, p  # every shape of the grid fits
        S, kc, R = p["S"], p["kc"], p["R"]
        assert kc * S >= NB and (S - 1) * kc < NB, p  # K covered, no empty slice
        assert kc <= max(1, 16 // p["nt"]), p  # one round of activation items per warp
        assert 1 <= R <= T and R * S <= max(SMS, S), p
        assert p["smem"] <= SMEM_MAX, p
        assert p["ws_floats"] == (S * M * N if S > 1 else 0), p
        in_kernel = S > 1 and M * S <= 16
        assert p["tickets"] == (R if in_kernel else 0), p


@needs_nvcc
def test_batched_plan_of_the_down_projection(plans):
    down = {p["M"]: p for p in plans["tcb"] if p["N"] == 4096 and p["K"] == 14336}
    one = down[1]
    assert (one["S"], one["R"], one["kc"], one["tickets"]) == (4, 38, 14, 38)
    sixteen = down[16]
    assert (sixteen["nt"], sixteen["S"], sixteen["tickets"]) == (4, 14, 0)


@needs_nvcc
def test_prefill_split(plans):
    for g in plans["gemm_split"]:
        tiles, K, full, ks = g["tiles"], g["K"], g["full"], g["ksplit"]
        assert 1 <= ks <= 16 and ks <= K // 256, g
        if tiles % SMS == 0:
            assert ks == 1 and full == tiles, g  # whole waves: nothing to split
        if ks > 1:
            assert full == tiles - tiles % SMS and full % SMS == 0, g  # only the tail wave splits
        else:
            assert full == tiles, g
    # a short tail of a long K is split; a nearly full wave is not
    d = {(g["tiles"], g["tok"], g["K"]): g for g in plans["gemm_split"]}
    assert d[(SMS + 8, 256, 14336)]["ksplit"] > 1
    assert d[(2 * SMS - 1, 256, 14336)]["ksplit"] == 1


@needs_nvcc
def test_prefill_tiles(plans):
    for g in plans["gemm_tiles"]:
        M, N, tok = g["M"], g["N"], g["tok"]
        assert g["tiles"] == -(-M // tok) * -(-N // 256), g
        assert g["smem"] <= SMEM_MAX, g


@needs_nvcc
def test_decode_kernel_shared_memory(plans):
    rows = {(r["K"], r["M"]): r for r in plans["tc_smem"]}
    for (K, M), r in rows.items():
        assert r["smem_16x2"] < r["smem_16x3"]
        if M > 1:
            assert rows[(K, M - 1)]["smem_16x2"] <= r["smem_16x2"]
    Ks = sorted({K for K, _ in rows})
    for M in range(1, 5):
        s = [rows[(K, M)]["smem_16x2"] for K in Ks]
        assert s == sorted(s)  # grows with K
    # the decode route takes every K <= 8192 for one row (checked with 3 slots)
    assert rows[(8192, 1)]["smem_16x3"] <= SMEM_MAX


@needs_nvcc
def test_fp32_gemv_plans(plans):
    for p in plans["gemv"]:
        fmt, N, K = p["fmt"], p["N"], p["K"]
        assert p["kchunks"] * p["ksplit"] == K // 64, p  # the row is cut into whole slices
        assert (K // 256) % p["ksplit"] == 0, p  # of whole 256-weight blocks
        assert p["kchunks"] <= 256 and p["threads"] <= 1024, p
        assert p["stage_rows"] == p["rg"] * p["rpg"] and p["rpg"] in (1, 2, 4), p
        assert 2 <= p["stages"] <= 16, p
        assert 1 <= p["row_slices"] <= N, p
        per_chunk = 36 if fmt == 12 else 68  # bytes of 64 weights: Q4_K, Q8_0
        assert p["slice_bytes"] == p["kchunks"] * per_chunk, p
        assert p["smem"] <= SMEM_MAX, p


@needs_nvcc
def test_m1_plans_cover_and_stay_in_bounds(plans):
    """The one-row decode kernel (gemv_m1.cu): for every plan, the index
    arithmetic of the kernel restated here -- slice s = b % S of KS
    super-blocks; item i = tiles [i*TS, (i+1)*TS) x the slice in NP passes of
    WS super-blocks, each pass one ring slot of W = WS*TS units of 2304 bytes;
    consumer warp w reads unit (w // WS, w % WS); CTA b1 of a slice takes items
    b1*F .. b1*F+F-1, then items G1*F + n from the counter, at most cap in all
    -- covers every (tile, super-block) exactly once, keeps every
    shared-memory index inside its array, sizes the counters and scratch to
    what is touched, and fits the shared memory of one CTA (two CTAs per SM
    with 8 consumer warps)."""
    rows = plans["m1"]
    assert rows
    for p in rows:
        T, NB, S, KS, WS, NP, TS, W = (p[k] for k in ("T", "NB", "S", "KS", "WS", "NP", "TS", "W"))
        maxw = p["maxw"]
        budget = 110 * 1024 if maxw == 8 else 226 * 1024
        tag = f"T={T} NB={NB} force={p['force']} maxw={maxw}"
        if p["nslot"] == 0:
            continue  # refused: the caller falls back to another kernel
        if p["force"]:
            assert S == p["force"], tag
        assert S * KS == NB and KS == WS * NP and 1 <= WS <= maxw, tag
        assert W == WS * TS and W <= maxw and TS in (1, 2, 4, 8), tag
        n_items, G1, F, cap = p["n_items"], p["G1"], p["F"], p["cap"]
        assert n_items == -(-T // TS), tag
        assert 1 <= G1 <= n_items and (G1 * S <= SMS or -(-n_items // G1) <= 16), tag
        assert 2 <= p["nslot"] <= 16, tag
        assert 1 <= F <= cap, tag
        # every item has a taker: the fixed shares plus cap per CTA cover them
        assert G1 * cap >= n_items, tag
        assert p["slot_bytes"] == W * 2304, tag
        assert p["smem"] == p["smem_check"] <= budget, tag
        assert p["ws_floats"] == (S * T * 16 if S > 1 else 0), tag
        assert p["tickets"] == 2 * S + (n_items if S > 1 else 0), tag
        # the largest byte a consumer lane reads in a slot: unit W-1, row 15,
        # bytes up to 144 of the row; a producer box u lands at u*WS*2304
        assert (W - 1) * 2304 + 15 * 144 + 144 <= p["slot_bytes"], tag
        assert (TS - 1) * WS * 2304 + WS * 2304 <= p["slot_bytes"], tag
        # fixed shares: items f*G1 + b1 below n_items, distinct over CTAs and
        # at most one apart in count (every CTA starts with its share)
        share = [sum(1 for f in range(F) if f * G1 + b < n_items) for b in range(G1)]
        fixed = {f * G1 + b for b in range(G1) for f in range(F) if f * G1 + b < n_items}
        assert len(fixed) == sum(share) == min(n_items, G1 * F), tag
        assert max(share) - min(share) <= 1, tag
        assert n_items * TS >= T > (n_items - 1) * TS, tag


@needs_nvcc
def test_m1_default_plans_for_llama_shapes(plans):
    """The default plans of the Llama-3.1-8B decode launches: gate/up (1792
    tiles), q/k/v (384) and o (256) whole K, one consumer warp per
    super-block (16), one pass; down (256 tiles of 56 super-blocks) in seven
    K slices of 8 super-blocks x 2 tiles (16 consumer warps), one pass."""
    by = {(p["T"], p["NB"]): p for p in plans["m1"] if p["force"] == 0 and p["maxw"] == 16}
    for T in (1792, 384, 256):
        assert by[(T, 16)]["S"] == 1 and by[(T, 16)]["W"] == 16 and by[(T, 16)]["NP"] == 1
    assert by[(256, 56)]["S"] == 7 and by[(256, 56)]["W"] == 16 and by[(256, 56)]["NP"] == 1


@needs_nvcc
def test_noalloc_shapes_split_k_and_refuse(plans):
    """The shapes tests/test_zz_no_alloc.py runs: at least one per format
    splits K (so the static scratch is written and read), every one of them
    fits, and the refused shape needs the scratch many times over (so the
    refusal does not hang on a planner detail)."""
    recs = {(r["fmt"], r["N"], r["K"]): r for r in plans["noalloc"]}
    for fmt in (12, 8):  # Q4_K, Q8_0
        run = [recs[(fmt, N, K)] for N, K in ((37, 2048), (3000, 4096), (5, 14336))]
        assert all(r["fits"] for r in run), run
        assert any(r["ksplit"] > 1 and r["need_floats"] > 0 for r in run), run
    big = recs[(12, 16384, 1 << 20)]
    assert not big["fits"] and big["need_floats"] >= 4 * big["have_floats"], big
