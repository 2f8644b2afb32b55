"""Benchmark: fused-dequant Q4_K decode GEMV over the Llama-3.1-8B linear
layers (32 layers x q,k,v,o,gate,up,down, batch 1), on GB300.

One step = one pass over all 32 layers' seven matrices: every weight byte of
the 3.93 GB Q4_K model is streamed once per step (the working set is 30x the
L2, so no flush is needed between steps).  q/k/v and gate/up share an input
and go out as grouped launches (128 launches per step, captured in a CUDA
graph with programmatic dependent launch).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-extras]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quantized_gguf_dequant_gb300 import synth  # noqa: E402

METRIC = "Q4_K dequant-GEMV HBM GB/s (% of peak); Q4_K prefill GEMM TFLOP/s (% peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SHAPES = synth.LLAMA8B_SHAPES
LAYERS = synth.LLAMA8B_LAYERS
SEED = 2026


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained")
            if hbm:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf or FALLBACK_BF16_TFLOPS),
                        "bf16_tflops_sustained": float(bfs or bf or FALLBACK_BF16_TFLOPS),
                        "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def layer_bytes(fmt):
    """Algorithmic bytes of one layer: every weight byte once, each distinct
    input vector once (q/k/v share one, gate/up share one), every output."""
    w = sum(N * synth.row_bytes(fmt, K) for _, N, K in SHAPES)
    x = 4 * (4096 + 4096 + 4096 + 14336)
    y = 4 * sum(N for _, N, _ in SHAPES)
    return w + x + y, w


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, pw = [], [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w_median": statistics.median(pw), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def time_oracle(seconds=10.0):
    """Oracle GEMV throughput over whole layers, generation excluded."""
    import oracle
    cores = os.cpu_count() or 1
    total_t = 0.0
    total_b = 0
    layers = 0
    while total_t < seconds and layers < LAYERS:
        for j, (name, N, K) in enumerate(SHAPES):
            w = synth.q4k_matrix(N, K, synth.layer_seed(SEED, layers, j))
            x = synth.activations(1, K, synth.layer_seed(SEED + 1, layers, j))[0]
            ts = time.perf_counter()
            oracle.gemv(synth.Q4_K, w, N, K, x, nthreads=cores)
            total_t += time.perf_counter() - ts
            total_b += N * synth.row_bytes(synth.Q4_K, K)
        layers += 1
    return {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{layers} of 32 Llama-3.1-8B layers (all 7 matrices, all rows), Q4_K, "
                      f"fp64 decode-then-dot, OpenMP over rows; {total_t:.1f} s of CPU time"}


# ------------------------------------------------------------------ GPU model

class Model:
    """32 layers of Q4_K (or Q8_0) weights resident on the device, with inputs
    and outputs laid out in two contiguous buffers."""

    def __init__(self, fmt, layers=LAYERS, device="cuda"):
        import torch
        import quantized_gguf_dequant_gb300 as q
        self.q = q
        self.fmt = fmt
        self.layers = []
        x_sizes = [4096, 4096, 4096, 14336]  # inputs of qkv, o, gate/up, down
        y_sizes = [N for _, N, _ in SHAPES]
        self.x_per_layer = sum(x_sizes)
        self.y_per_layer = sum(y_sizes)
        self.x_all = torch.empty(layers * self.x_per_layer, dtype=torch.float32, device=device)
        self.y_all = torch.empty(layers * self.y_per_layer, dtype=torch.float32, device=device)
        xs = synth.activations(layers, self.x_per_layer, SEED + 7)
        self.x_host = torch.from_numpy(xs.reshape(-1)).pin_memory()
        self.x_all.copy_(self.x_host)
        self.y_host = torch.empty(layers * self.y_per_layer, dtype=torch.float32).pin_memory()
        for L in range(layers):
            mats = []
            for j, (name, N, K) in enumerate(SHAPES):
                w = synth.matrix(fmt, N, K, synth.layer_seed(SEED, L, j))
                mats.append(q.Matrix(fmt, N, K, torch.from_numpy(w).to(device)))
            xo = L * self.x_per_layer
            xv = []
            for s in x_sizes:
                xv.append(self.x_all[xo:xo + s])
                xo += s
            yo = L * self.y_per_layer
            yv = []
            for s in y_sizes:
                yv.append(self.y_all[yo:yo + s])
                yo += s
            self.layers.append((mats, xv, yv))
        torch.cuda.synchronize()

    def step(self, grouped=True):
        q = self.q
        for mats, xv, yv in self.layers:
            mq, mk, mv, mo, mg, mu, md = mats
            if grouped:
                q.gemv_group([mq.h, mk.h, mv.h], xv[0], yv[0:3])
                q.gemv(mo.h, xv[1], yv[3])
                q.gemv_group([mg.h, mu.h], xv[2], yv[4:6])
            else:
                q.gemv(mq.h, xv[0], yv[0])
                q.gemv(mk.h, xv[0], yv[1])
                q.gemv(mv.h, xv[0], yv[2])
                q.gemv(mo.h, xv[1], yv[3])
                q.gemv(mg.h, xv[2], yv[4])
                q.gemv(mu.h, xv[2], yv[5])
            q.gemv(md.h, xv[3], yv[6])

    def step_subset(self, which):
        """Only the launches of one kernel family: 'short' = the K=4096
        projections (q/k/v group, o, gate/up group), 'long' = down (K=14336)."""
        q = self.q
        for mats, xv, yv in self.layers:
            mq, mk, mv, mo, mg, mu, md = mats
            if which == "short":
                q.gemv_group([mq.h, mk.h, mv.h], xv[0], yv[0:3])
                q.gemv(mo.h, xv[1], yv[3])
                q.gemv_group([mg.h, mu.h], xv[2], yv[4:6])
            else:
                q.gemv(md.h, xv[3], yv[6])

    def q8k_step(self, which="all", fused=False):
        """The decode step on the integer-dot variant: each distinct input
        quantized to Q8_K once (qmm_quantize_q8_k), then qmm_gemv_q8k_group
        (q/k/v, gate/up) and qmm_gemv_q8k (o, down); fused: the quantization
        inside each GEMV launch (qmm_gemv_q8k_fused[_group]).  which: 'all',
        'short' (the K=4096 launches with their quantizations) or 'long'
        (down)."""
        import torch
        q = self.q
        if fused:
            for mats, xv, yv in self.layers:
                mq, mk, mv, mo, mg, mu, md = mats
                if which in ("all", "short"):
                    q.gemv_q8k_fused_group([mq.h, mk.h, mv.h], xv[0], yv[0:3])
                    q.gemv_q8k_fused(mo.h, xv[1], yv[3])
                    q.gemv_q8k_fused_group([mg.h, mu.h], xv[2], yv[4:6])
                if which in ("all", "long"):
                    q.gemv_q8k_fused(md.h, xv[3], yv[6])
            return
        if getattr(self, "xq", None) is None:
            sizes = [4096, 4096, 4096, 14336]
            self.xq = [[torch.empty(k // 256 * q.Q8_K_BLOCK, dtype=torch.uint8,
                                    device=self.x_all.device) for k in sizes]
                       for _ in self.layers]
        for L, (mats, xv, yv) in enumerate(self.layers):
            mq, mk, mv, mo, mg, mu, md = mats
            xq = self.xq[L]
            if which in ("all", "short"):
                q.quantize_q8_k(xv[0], 4096, xq[0])
                q.gemv_q8k_group([mq.h, mk.h, mv.h], xq[0], yv[0:3])
                q.quantize_q8_k(xv[1], 4096, xq[1])
                q.gemv_q8k(mo.h, xq[1], yv[3])
                q.quantize_q8_k(xv[2], 4096, xq[2])
                q.gemv_q8k_group([mg.h, mu.h], xq[2], yv[4:6])
            if which in ("all", "long"):
                q.quantize_q8_k(xv[3], 14336, xq[3])
                q.gemv_q8k(md.h, xq[3], yv[6])

    def ffn_step(self, fused=True):
        """The dense SwiGLU FFN of every layer (gate, up, down): qmm_ffn_decode,
        or the grouped gate/up GEMV, qmm_swiglu and the down GEMV as separate
        calls.  h lands in the gate's output slot."""
        q = self.q
        for mats, xv, yv in self.layers:
            mg, mu, md = mats[4], mats[5], mats[6]
            if fused:
                q.ffn_decode(mg.h, mu.h, md.h, xv[2], yv[4], yv[6])
            else:
                q.gemv_group([mg.h, mu.h], xv[2], yv[4:6])
                q.swiglu(yv[4], yv[5], yv[4], yv[4].numel())
                q.gemv(md.h, yv[4], yv[6])

    def ffn_bytes(self):
        """Algorithmic bytes of ffn_step: gate/up/down weights once, x, h
        written and read once, y."""
        w = sum(N * synth.row_bytes(self.fmt, K) for name, N, K in SHAPES
                if name in ("gate", "up", "down"))
        return (w + 4 * (4096 + 2 * 14336 + 4096)) * len(self.layers)

    def launches(self, grouped=True):
        return len(self.layers) * (4 if grouped else 7)

    def close(self):
        for mats, _, _ in self.layers:
            for m in mats:
                m.close()


class BatchedModel:
    """Continuous-batching decode: the Llama-3.1-8B Q4_K matrices of a Model
    applied to M activation rows per call (one read of the weights for all M)."""

    def __init__(self, model, M_max=16, device="cuda"):
        import torch
        self.model = model
        self.M_max = M_max
        x_sizes = [4096, 4096, 4096, 14336]
        nl = len(model.layers)
        xs = synth.activations(nl * M_max, sum(x_sizes), SEED + 11)
        self.X = torch.from_numpy(xs).to(device).view(nl, M_max, sum(x_sizes))
        self.xoff = [0, 4096, 8192, 12288]
        self.kin = [0, 0, 0, 1, 2, 2, 3]  # which input each matrix reads
        self.Y = [torch.empty((M_max, N), dtype=torch.float32, device=device)
                  for _, N, _ in SHAPES]

    def step(self, M):
        q = self.model.q
        for L, (mats, _, _) in enumerate(self.model.layers):
            XL = self.X[L]
            for j, m in enumerate(mats):
                i = self.kin[j]
                x = XL[:, self.xoff[i]:]
                q.gemv_batched(m.h, x.data_ptr(), M, XL.stride(0), self.Y[j], self.Y[j].stride(0))

    def bytes_per_step(self, M):
        w = sum(N * synth.row_bytes(synth.Q4_K, K) for _, N, K in SHAPES)
        x = 4 * M * (4096 + 4096 + 4096 + 14336)
        y = 4 * M * sum(N for _, N, _ in SHAPES)
        return (w + x + y) * len(self.model.layers)


class MoeModel:
    """OLMoE-1B-7B expert layers: 64 experts, d_model 2048, d_ff 1024, Q4_K,
    32 tokens routed top-8 by a seeded softmax; one step runs every layer's
    whole expert FFN (bucket, gate+up, SwiGLU, down, combine)."""

    def __init__(self, layers=16, T=32, device="cuda", fmt=synth.Q4_K):
        import torch
        import quantized_gguf_dequant_gb300 as q
        self.q = q
        E, dm, dff, k = synth.OLMOE_EXPERTS, synth.OLMOE_D_MODEL, synth.OLMOE_D_FF, synth.OLMOE_TOP_K
        self.E, self.T, self.k, self.dm, self.dff = E, T, k, dm, dff
        self.layers = []
        self.active_bytes = 0
        # gate, up (dff rows of dm) and down (dm rows of dff)
        per_expert = 2 * dff * synth.row_bytes(fmt, dm) + dm * synth.row_bytes(fmt, dff)
        for L in range(layers):
            hs = []
            for j, (N, K) in enumerate(((E * dff, dm), (E * dff, dm), (E * dm, dff))):
                w = synth.matrix(fmt, N, K, synth.layer_seed(SEED + 100, L, j))
                hs.append(q.Matrix(fmt, N, K, torch.from_numpy(w).to(device)))
            ids, r = synth.router(T, E, k, synth.layer_seed(SEED + 200, L, 0))
            X = synth.activations(T, dm, synth.layer_seed(SEED + 300, L, 0))
            self.active_bytes += len(np.unique(ids)) * per_expert
            self.layers.append((hs, torch.from_numpy(ids).to(device), torch.from_numpy(r).to(device),
                                torch.from_numpy(X).to(device),
                                torch.empty((T, dm), dtype=torch.float32, device=device)))
        torch.cuda.synchronize()

    def step(self):
        q = self.q
        for hs, ids, r, X, Y in self.layers:
            q.moe_ffn(hs[0].h, hs[1].h, hs[2].h, self.E, ids, self.T, self.k, X, r, Y)

    def bytes_per_step(self):
        xy = 2 * 4 * self.T * self.dm + 2 * 4 * self.T * self.k  # X, Y, ids, r
        return self.active_bytes + xy * len(self.layers)

    def close(self):
        for hs, *_ in self.layers:
            for h in hs:
                h.close()


class PrefillModel:
    """Prefill: the seven Llama-3.1-8B Q4_K matrices of `layers` layers applied
    to M bf16 tokens each (qmm_gemm per matrix; Y fp32)."""

    def __init__(self, M, layers=4, device="cuda"):
        import torch
        import quantized_gguf_dequant_gb300 as q
        self.q, self.M = q, M
        self.mats = []
        for L in range(layers):
            row = []
            for j, (name, N, K) in enumerate(SHAPES):
                w = synth.q4k_matrix(N, K, synth.layer_seed(SEED + 400, L, j))
                row.append(q.Matrix(synth.Q4_K, N, K, torch.from_numpy(w).to(device)))
            self.mats.append(row)
        self.X = {K: torch.from_numpy(synth.activations_bf16(M, K, SEED + K).view(np.int16)).to(device)
                  for K in sorted({K for _, _, K in SHAPES})}
        self.Y = [torch.empty((M, N), dtype=torch.float32, device=device) for _, N, _ in SHAPES]
        torch.cuda.synchronize()

    def step(self):
        q = self.q
        for row in self.mats:
            mq, mk, mv, mo, mg, mu, md = row
            q.gemm_group([mq.h, mk.h, mv.h], self.X[4096], self.M, self.Y[0:3])
            mo.gemm(self.X[4096], self.Y[3])
            q.gemm_group([mg.h, mu.h], self.X[4096], self.M, self.Y[4:6])
            md.gemm(self.X[14336], self.Y[6])

    def flops_per_step(self):
        return 2.0 * self.M * sum(N * K for _, N, K in SHAPES) * len(self.mats)

    def close(self):
        for row in self.mats:
            for m in row:
                m.close()


def small_matrix_extra(pk):
    """The 1024 x 1024 Q4_K matrix alone: (i) single-call latency with L2
    flushed before every call (a 256 MB write between calls), median of 21;
    (ii) throughput over 512 distinct copies (302 MB > L2) in one graph."""
    import torch
    import quantized_gguf_dequant_gb300 as q
    N = K = 1024
    copies = 512
    mats = [q.Matrix(synth.Q4_K, N, K, torch.from_numpy(synth.q4k_matrix(N, K, 7000 + i)).cuda())
            for i in range(copies)]
    x = torch.from_numpy(synth.activations(1, K, 7)[0]).cuda()
    ys = torch.empty((copies, N), dtype=torch.float32, device="cuda")
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
    wbytes = N * synth.row_bytes(synth.Q4_K, K)
    lat = []
    for i in range(24):
        flush.fill_(float(i))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        q.gemv(mats[i].h, x, ys[i])
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            lat.append(e0.elapsed_time(e1) * 1e3)
    # The same harness around a one-element add (the floor of any kernel launch
    # between two events after the flush)
    one = torch.zeros(1, device="cuda")
    floor = []
    for i in range(24):
        flush.fill_(float(i))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        one.add_(1.0)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            floor.append(e0.elapsed_time(e1) * 1e3)
    # In a graph: (flush + call) x 20 minus flush x 20, per call -- the call's
    # added time with L2 flushed, without the events' own resolution; the same
    # for a 590 KB device copy.
    src = torch.empty(wbytes // 4, dtype=torch.float32, device="cuda")
    dst = torch.empty_like(src)
    t_fl, _ = time_graph(lambda: [flush.fill_(1.0) for _ in range(20)], 3, 3, 1)
    t_gv, _ = time_graph(lambda: [(flush.fill_(1.0), q.gemv(mats[0].h, x, ys[0])) for _ in range(20)], 3, 3, 1)
    t_cp, _ = time_graph(lambda: [(flush.fill_(1.0), dst.copy_(src)) for _ in range(20)], 3, 3, 1)
    ms, _ = time_graph(lambda: [q.gemv(m.h, x, ys[i]) for i, m in enumerate(mats)], 5, 3, 1)
    tput = copies * (wbytes + 4 * K + 4 * N) / (ms * 1e-3) / 1e9
    for m in mats:
        m.close()
    del flush
    return {"latency_us_median": statistics.median(lat), "latency_us_min": min(lat),
            "one_element_kernel_latency_us_median": statistics.median(floor),
            "graph_added_us_per_call": (t_gv - t_fl) * 1e3 / 20,
            "graph_added_us_per_590kb_copy": (t_cp - t_fl) * 1e3 / 20,
            "rotating_gbs": tput, "rotating_frac_of_peak": tput / pk["hbm_gbs"],
            "note": "qmm_gemv on a 1024 x 1024 Q4_K matrix (589,824 B): latency of one call with "
                    "L2 flushed (CUDA events around the call; the same harness around a one-element "
                    "add kernel gives its floor), the time one call adds to a graph of flushes, "
                    "beside a 590 KB device copy, and 512 distinct copies in one CUDA graph "
                    "(weights > L2)"}


def launches_of(fn):
    """Kernels the library launches for one call of fn (counted by the
    library itself; run eagerly, outside any capture)."""
    import torch
    import quantized_gguf_dequant_gb300 as q
    c0 = q.launch_count()
    fn()
    torch.cuda.synchronize()
    return q.launch_count() - c0


def time_graph(fn, steps, warmup, world, sampler_index=None):
    """Capture fn into a CUDA graph, replay warmup + steps; returns (ms/step,
    clocks summary)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the launch path outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    clocks = None
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    if sampler:
        sampler.__enter__()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
        clocks = sampler.summary()
    ms = e0.elapsed_time(e1) / steps
    ms = max_over_ranks(world, ms)
    del g
    return ms, clocks


def time_graph_stats(fn, reps, warmup, world):
    """Capture fn into a CUDA graph, replay warmup times, then reps times with
    an event pair around each replay; returns {median_ms, min_ms, mean_ms,
    reps} over the replays (max over ranks)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warmup):
        g.replay()
    barrier(world)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    barrier(world)
    t = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
    del g
    return {"median_ms": max_over_ranks(world, statistics.median(t)),
            "min_ms": max_over_ranks(world, min(t)),
            "mean_ms": max_over_ranks(world, sum(t) / reps), "reps": reps}


def time_eager(fn, steps, warmup, world):
    """Direct launches (no graph); used for profiling runs."""
    import torch
    for _ in range(warmup):
        fn()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(world, e0.elapsed_time(e1) / steps), None


def time_e2e(model, steps, warmup, world):
    """Same metric through the public API with host buffers: per step, copy
    every input vector host->device (pinned), issue the layer calls, copy every
    output back and wait for it."""
    import torch
    stream = torch.cuda.current_stream()

    def one():
        model.x_all.copy_(model.x_host, non_blocking=True)
        model.step(grouped=True)
        model.y_host.copy_(model.y_all, non_blocking=True)
        stream.synchronize()

    for _ in range(warmup):
        one()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    barrier(world)
    ms = max_over_ranks(world, dt * 1e3 / steps)
    return ms, model.x_host.numel() * 4, model.y_host.numel() * 4


# ------------------------------------------------------------------ traffic

def recorded_traffic(kernel_key):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if it
    was taken on the kernel sources as they are now (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(kernel_key)
        h = hashlib.sha256()
        for src in rec["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest()[:16] != rec["sources_sha"]:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ main arms

def run_ours(args, world, rank, local):
    import torch
    torch.cuda.set_device(local)
    pk = peaks()
    nl = args.layers
    q4 = Model(synth.Q4_K, layers=nl)
    bytes_layer, wbytes_layer = layer_bytes(synth.Q4_K)
    step_bytes = bytes_layer * nl
    if args.graph:
        ms, clocks = time_graph(lambda: q4.step(True), args.steps, args.warmup, world,
                                sampler_index=local)
    else:
        ms, clocks = time_eager(lambda: q4.step(True), args.steps, args.warmup, world)
    gbs = step_bytes / (ms * 1e-3) / 1e9 * world
    per_gpu = step_bytes / (ms * 1e-3) / 1e9
    launches_per_step = launches_of(lambda: q4.step(True))
    launches = launches_per_step * args.steps
    # Each family of launches timed on its own (same graph + PDL set-up): the
    # K=4096 projections (q/k/v group, o, gate/up group) and down (K=14336,
    # seven K slices), all on the one-row decode kernel.
    fam = {}
    wb = {s_: 0 for s_ in ("short", "long")}
    for name, N, K in SHAPES:
        wb["long" if K > 8192 else "short"] += N * synth.row_bytes(synth.Q4_K, K)
    xy = {"short": 4 * (3 * 4096 + 4096 + 1024 * 2 + 4096 + 14336 * 2),
          "long": 4 * (14336 + 4096)}
    for which, kname in (("short", "gemv_m1_kernel"), ("long", "gemv_m1_kernel")):
        st = time_graph_stats(lambda: q4.step_subset(which), max(20, args.steps // 4), args.warmup,
                              world)
        ms_f = st["median_ms"]
        b = (wb[which] + xy[which]) * nl
        fam[which] = {"kernel": kname, "ms_per_step": ms_f, "min_ms": st["min_ms"],
                      "reps": st["reps"], "bytes_per_step": b,
                      "launches_per_step": launches_of(lambda: q4.step_subset(which)),
                      "gbs": b / (ms_f * 1e-3) / 1e9}
    extras = {}
    e2e = None
    if args.e2e:
        e2e_ms, h2d, d2h = time_e2e(q4, max(10, min(args.steps // 10, 300)), 3, world)
        e2e = {"value": step_bytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms,
               "how": "per step: pinned H2D of every input vector, the qmm_gemv / "
                      "qmm_gemv_group calls through the binding (no graph), D2H of every "
                      "output, stream sync"}
    if args.extras:
        st_u = time_graph_stats(lambda: q4.step(False), max(20, args.steps // 4), args.warmup, world)
        ms_u = st_u["median_ms"]
        extras["q4k_decode_ungrouped"] = {
            "value": step_bytes / (ms_u * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_u,
            "min_ms": st_u["min_ms"], "reps": st_u["reps"],
            "launches_per_step": launches_of(lambda: q4.step(False)),
            "frac_of_peak": step_bytes / (ms_u * 1e-3) / 1e9 / pk["hbm_gbs"]}
    if args.extras:
        # The integer-dot variant on the same 32-layer step: every distinct
        # input quantized to Q8_K once, then the integer GEMVs.
        st_q = time_graph_stats(lambda: q4.q8k_step("all"), max(20, args.steps // 4), args.warmup,
                                world)
        ms_q = st_q["median_ms"]
        extras["q4k_decode_q8k_integer"] = {
            "value": step_bytes / (ms_q * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_q,
            "min_ms": st_q["min_ms"], "reps": st_q["reps"],
            "launches_per_step": launches_of(lambda: q4.q8k_step("all")),
            "frac_of_peak": step_bytes / (ms_q * 1e-3) / 1e9 / pk["hbm_gbs"],
            "f32_over_q8k_time": ms / ms_q,
            "note": "opt-in Q8_K activations + dp4a integer dot (qmm_quantize_q8_k, "
                    "qmm_gemv_q8k[_group]); bytes counted as for the f32 step (weights once, "
                    "f32 inputs once, outputs); drift vs f32 bounded by sum |w| |d|/2 per block"}
        st_f = time_graph_stats(lambda: q4.q8k_step("all", fused=True), max(20, args.steps // 4),
                                args.warmup, world)
        ms_f = st_f["median_ms"]
        extras["q4k_decode_q8k_integer_fused"] = {
            "value": step_bytes / (ms_f * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_f,
            "min_ms": st_f["min_ms"], "reps": st_f["reps"],
            "launches_per_step": launches_of(lambda: q4.q8k_step("all", fused=True)),
            "frac_of_peak": step_bytes / (ms_f * 1e-3) / 1e9 / pk["hbm_gbs"],
            "f32_over_q8k_time": ms / ms_f,
            "note": "the same integer-dot step with the Q8_K quantization inside each GEMV "
                    "launch (qmm_gemv_q8k_fused[_group]; bitwise equal results)"}
    if args.extras:
        bm = BatchedModel(q4)
        sweep = {}
        for M in (1, 2, 4, 8, 16):
            st_b = time_graph_stats(lambda: bm.step(M), max(20, args.steps // 8), args.warmup, world)
            ms_b = st_b["median_ms"]
            b = bm.bytes_per_step(M)
            sweep[str(M)] = {"ms_per_step": ms_b, "min_ms": st_b["min_ms"], "reps": st_b["reps"],
                             "gbs": b / (ms_b * 1e-3) / 1e9,
                             "frac_of_peak": b / (ms_b * 1e-3) / 1e9 / pk["hbm_gbs"],
                             "tokens_per_s": M / (ms_b * 1e-3),
                             "launches_per_step": launches_of(lambda: bm.step(M))}
        extras["q4k_batched_decode"] = {
            "unit": "GB/s", "by_M": sweep,
            "note": "qmm_gemv_batched on every matrix of every layer, M activation rows per "
                    "call; bytes = weights once + M input rows + M output rows"}
        del bm
    if args.extras:
        fb = q4.ffn_bytes()
        ffn = {}
        for fused in (True, False):
            st_f = time_graph_stats(lambda: q4.ffn_step(fused), max(20, args.steps // 4), args.warmup,
                                   world)
            ms_f = st_f["median_ms"]
            ffn["fused" if fused else "separate"] = {
                "ms_per_step": ms_f, "min_ms": st_f["min_ms"], "reps": st_f["reps"],
                "gbs": fb / (ms_f * 1e-3) / 1e9,
                "frac_of_peak": fb / (ms_f * 1e-3) / 1e9 / pk["hbm_gbs"],
                "launches_per_step": launches_of(lambda: q4.ffn_step(fused))}
        extras["q4k_dense_ffn_decode"] = {
            "unit": "GB/s", "bytes_per_step": fb, **ffn,
            "note": "the Llama-3.1-8B SwiGLU FFN of every layer for one token: qmm_ffn_decode "
                    "(gate and up in one decode-kernel launch, their tiles interleaved, SwiGLU "
                    "in its output phase, then down) against the grouped gate/up GEMV, "
                    "qmm_swiglu and the down GEMV as separate calls"}
    q4.close()
    del q4
    torch.cuda.empty_cache()
    if args.extras:
        extras["q4k_1024x1024"] = small_matrix_extra(pk)
        torch.cuda.empty_cache()
    if args.extras:
        mo = MoeModel()
        st_m = time_graph_stats(mo.step, max(20, args.steps // 4), args.warmup, world)
        ms_m = st_m["median_ms"]
        bm_ = mo.bytes_per_step()
        extras["olmoe_moe_ffn"] = {
            "value": bm_ / (ms_m * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_m,
            "min_ms": st_m["min_ms"], "reps": st_m["reps"],
            "bytes_per_step": bm_, "layers": len(mo.layers), "tokens": mo.T,
            "frac_of_peak": bm_ / (ms_m * 1e-3) / 1e9 / pk["hbm_gbs"],
            "us_per_layer": ms_m * 1e3 / len(mo.layers), "launches_per_step": launches_of(mo.step),
            "note": "qmm_moe_ffn per layer (bucket, gate+up, SwiGLU, down, combine); bytes = "
                    "the Q4_K gate/up/down bytes of every expert some token picked, plus X, Y, "
                    "ids and routing weights; 16 layers = 3.6 GB of experts > L2"}
        mo.close()
        del mo
        torch.cuda.empty_cache()
        mo = MoeModel(fmt=synth.Q8_0)
        st_m = time_graph_stats(mo.step, max(20, args.steps // 4), args.warmup, world)
        ms_m = st_m["median_ms"]
        bm_ = mo.bytes_per_step()
        extras["olmoe_moe_ffn_q8_0"] = {
            "value": bm_ / (ms_m * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_m,
            "min_ms": st_m["min_ms"], "reps": st_m["reps"],
            "bytes_per_step": bm_, "layers": len(mo.layers), "tokens": mo.T,
            "frac_of_peak": bm_ / (ms_m * 1e-3) / 1e9 / pk["hbm_gbs"],
            "us_per_layer": ms_m * 1e3 / len(mo.layers), "launches_per_step": launches_of(mo.step),
            "note": "the same OLMoE expert FFN with Q8_0 experts (moe_q8_kernel for gate+up "
                    "with SwiGLU, and for down); 16 layers = 6.8 GB of experts"}
        mo.close()
        del mo
        torch.cuda.empty_cache()
    if args.extras:
        pre = {}
        for M in (512, 2048):
            pm = PrefillModel(M)
            st_p = time_graph_stats(pm.step, max(20, args.steps // 40), args.warmup, world)
            ms_p = st_p["median_ms"]
            fl = pm.flops_per_step()
            tf = fl / (ms_p * 1e-3) / 1e12
            pre[str(M)] = {"ms_per_step": ms_p, "min_ms": st_p["min_ms"], "reps": st_p["reps"],
                           "tflops": tf, "tflops_at_min": fl / (st_p["min_ms"] * 1e-3) / 1e12,
                           "frac_of_peak": tf / pk["bf16_tflops"],
                           "launches_per_step": launches_of(pm.step)}
            pm.close()
            del pm
            torch.cuda.empty_cache()
        extras["q4k_prefill_gemm"] = {
            "unit": "TFLOP/s", "by_M": pre,
            "roofline": {"bound": "tensor", "kernel": "gemm_q4k_kernel",
                         "achieved": pre["2048"]["tflops"], "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": pre["2048"]["tflops"] / pk["bf16_tflops"],
                         "peak_source": pk["source"], "traffic": recorded_traffic("gemm_q4k_kernel")},
            "note": "the 7 Llama-3.1-8B matrices of 4 layers (491 MB of Q4_K weights > L2) as "
                    "qmm_gemm_group (q/k/v, gate/up share X) and qmm_gemm (o, down), bf16 X of M "
                    "tokens, fp32 Y; flops = 2*M*N*K; peak = bf16 "
                    "dense (burst figure: each GEMM is a separate launch of tens to hundreds "
                    "of microseconds)"}
    if args.extras:
        q8 = Model(synth.Q8_0, layers=nl)
        b8, _ = layer_bytes(synth.Q8_0)
        st8 = time_graph_stats(lambda: q8.step(True), max(20, args.steps // 4), args.warmup, world)
        ms8 = st8["median_ms"]
        extras["q8_0_decode"] = {
            "value": b8 * nl / (ms8 * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms8,
            "min_ms": st8["min_ms"], "reps": st8["reps"],
            "bytes_per_step": b8 * nl,
            "frac_of_peak": b8 * nl / (ms8 * 1e-3) / 1e9 / pk["hbm_gbs"]}
        q8.close()
        del q8
        torch.cuda.empty_cache()
    if args.extras:
        # Context for the fusion itself: the same 4-layer Q4_K decode step done
        # the unfused way -- each matrix decoded to a bf16 buffer in HBM
        # (qmm_dequantize_bf16), then a cuBLAS bf16 GEMV through torch.matmul
        # (x given in bf16 already).  Not a product path; a reported baseline.
        try:
            mu = Model(synth.Q4_K, layers=4)
            kin = [0, 0, 0, 1, 2, 2, 3]
            xbs = [[x.to(torch.bfloat16) for x in xv] for _, xv, _ in mu.layers]
            ybs = [[torch.empty(N, dtype=torch.bfloat16, device="cuda") for _, N, _ in SHAPES]
                   for _ in mu.layers]
            wbuf = torch.empty(max(N * K for _, N, K in SHAPES), dtype=torch.int16, device="cuda")
            q = mu.q

            def unfused_step():
                for L, (mats, _, _) in enumerate(mu.layers):
                    for j, m in enumerate(mats):
                        q.dequantize_bf16(m.h, 0, m.N, wbuf)
                        W = wbuf[:m.N * m.K].view(torch.bfloat16).view(m.N, m.K)
                        torch.matmul(W, xbs[L][kin[j]], out=ybs[L][j])

            nsteps = max(3, args.steps // 20)
            st_un = time_graph_stats(unfused_step, max(20, nsteps), args.warmup, world)
            st_fu = time_graph_stats(lambda: mu.step(True), max(20, nsteps), args.warmup, world)
            ms_un, ms_fu = st_un["median_ms"], st_fu["median_ms"]
            b4, _ = layer_bytes(synth.Q4_K)
            extras["unfused_torch_baseline"] = {
                "layers": 4, "ms_per_step_unfused": ms_un, "ms_per_step_fused": ms_fu,
                "min_ms_unfused": st_un["min_ms"], "min_ms_fused": st_fu["min_ms"],
                "reps": st_un["reps"],
                "unfused_over_fused": ms_un / ms_fu,
                "gbs_unfused": b4 * 4 / (ms_un * 1e-3) / 1e9, "gbs_fused": b4 * 4 / (ms_fu * 1e-3) / 1e9,
                "unit": "GB/s of quantized algorithmic bytes",
                "note": "decode to a bf16 buffer (qmm_dequantize_bf16) then torch.matmul (cuBLAS) per "
                        "matrix, against the fused path on the same 4 layers"}
            mu.close()
            del mu, wbuf, xbs, ybs
        except Exception as e:  # a secondary line: report, do not lose the run
            extras["unfused_torch_baseline"] = {"error": f"{type(e).__name__}: {e}"}
        try:
            torch.cuda.empty_cache()
        except Exception:
            pass
    if args.extras:
        # The further block formats on the same decode step (4 layers, > L2),
        # through the plain one-warp-per-row decode GEMV.
        fx = {}
        for fname, fcode in (("Q5_K", synth.Q5_K), ("Q6_K", synth.Q6_K), ("IQ4_NL", synth.IQ4_NL)):
            try:
                mf = Model(fcode, layers=4)
                bf, _ = layer_bytes(fcode)
                st_x = time_graph_stats(lambda: mf.step(True), max(20, args.steps // 8),
                                        args.warmup, world)
                ms_x = st_x["median_ms"]
                fx[fname] = {"ms_per_step": ms_x, "min_ms": st_x["min_ms"], "reps": st_x["reps"],
                             "layers": 4, "bytes_per_step": bf * 4,
                             "gbs": bf * 4 / (ms_x * 1e-3) / 1e9,
                             "frac_of_peak": bf * 4 / (ms_x * 1e-3) / 1e9 / pk["hbm_gbs"]}
                mf.close()
                del mf
            except Exception as e:  # a secondary line: report, do not lose the run
                fx[fname] = {"error": f"{type(e).__name__}: {e}"}
            try:
                torch.cuda.empty_cache()
            except Exception:
                pass
        extras["extra_formats_decode"] = dict(
            fx, unit="GB/s",
            note="Llama-3.1-8B decode step, 4 layers (graph, PDL), the weights in each further "
                 "format, through the library's default route: the tensor-core decode kernel "
                 "(gemv_m1_kernel<Q5_K / Q6_K / IQ4_NL>, codes as exact fp16 subnormals)")

    # Every launch of the step is the one-row decode kernel, so its average
    # launch is the step's: algorithmic bytes per launch = step bytes / launches,
    # launch duration = the step's device time / launches.
    kname = "gemv_m1_kernel"
    assert all(f["kernel"] == kname for f in fam.values())
    traffic = recorded_traffic(kname)
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(decode_config(nl, world), launches_per_step=launches_per_step),
        "roofline": {"bound": "hbm", "achieved": per_gpu, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": per_gpu / pk["hbm_gbs"], "traffic": traffic,
                     "kernel": kname, "peak_source": pk["source"],
                     "launches_per_step": launches_per_step,
                     "algorithmic_bytes_per_launch": step_bytes / launches_per_step,
                     "launch_ms": ms / launches_per_step,
                     "note": "the step is launches of this one kernel only (100% of the step's "
                             "device time); achieved = algorithmic bytes per launch (weights "
                             "once, inputs once, outputs; mean over the step's launch mix) / "
                             "mean launch duration (CUDA events over the timed region / "
                             "launches); traffic = ncu DRAM bytes per launch over the same mix, "
                             "from profiles/traffic.json when taken on the current source"},
        "kernels": fam,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "extras": extras,
    }
    return line


def run_only(args, world, local):
    """One secondary workload alone (for profiling runs)."""
    import torch
    torch.cuda.set_device(local)
    timer = time_graph if args.graph else time_eager
    if args.only == "prefill":
        pm = PrefillModel(args.prefill_m, layers=args.layers)
        ms, _ = timer(pm.step, args.steps, args.warmup, world)
        tf = pm.flops_per_step() / (ms * 1e-3) / 1e12
        pm.close()
        return {"workload": f"prefill GEMM M={args.prefill_m}, {args.layers} layers", "ms_per_step": ms,
                "tflops": tf}
    if args.only == "q8":
        q8 = Model(synth.Q8_0, layers=args.layers)
        b8, _ = layer_bytes(synth.Q8_0)
        ms, _ = timer(lambda: q8.step(True), args.steps, args.warmup, world)
        q8.close()
        return {"workload": f"Llama-3.1-8B Q8_0 decode, {args.layers} layers", "ms_per_step": ms,
                "gbs": b8 * args.layers / (ms * 1e-3) / 1e9}
    if args.only == "tall":
        # The decode kernel's steady streaming rate: one Q4_K GEMV on a
        # 131072 x 4096 matrix (302 MB), where a launch's fixed cost is a few
        # percent of its time.
        import quantized_gguf_dequant_gb300 as q
        N, K = 131072, 4096
        w = torch.from_numpy(synth.q4k_matrix(N, K, SEED + 900)).cuda()
        m = q.Matrix(synth.Q4_K, N, K, w)
        x = torch.from_numpy(synth.activations(1, K, SEED + 901)[0]).cuda()
        y = torch.empty(N, dtype=torch.float32, device="cuda")
        ms, _ = timer(lambda: q.gemv(m.h, x, y), args.steps, args.warmup, world)
        nbytes = N * synth.row_bytes(synth.Q4_K, K) + 4 * K + 4 * N
        m.close()
        return {"workload": "Q4_K GEMV 131072 x 4096 (302 MB), one launch", "ms_per_step": ms,
                "gbs": nbytes / (ms * 1e-3) / 1e9}
    if args.only == "ffn":
        q4 = Model(synth.Q4_K, layers=args.layers)
        out = {"workload": f"Llama-3.1-8B dense FFN decode, {args.layers} layers"}
        for fused in (True, False):
            ms, _ = timer(lambda: q4.ffn_step(fused), args.steps, args.warmup, world)
            out["fused" if fused else "separate"] = {
                "ms_per_step": ms, "gbs": q4.ffn_bytes() / (ms * 1e-3) / 1e9}
        q4.close()
        return out
    if args.only == "batched":
        q4 = Model(synth.Q4_K, layers=args.layers)
        bm = BatchedModel(q4)
        out = {"workload": f"batched Q4_K decode, {args.layers} layers"}
        for M in (1, 2, 4, 8, 16):
            ms, _ = timer(lambda: bm.step(M), args.steps, args.warmup, world)
            out[str(M)] = {"ms_per_step": ms, "gbs": bm.bytes_per_step(M) / (ms * 1e-3) / 1e9}
        q4.close()
        return out
    mo = MoeModel(layers=args.layers)
    ms, _ = timer(mo.step, args.steps, args.warmup, world)
    gbs = mo.bytes_per_step() / (ms * 1e-3) / 1e9
    mo.close()
    return {"workload": f"OLMoE expert FFN, {args.layers} layers", "ms_per_step": ms, "gbs": gbs}


def decode_config(nl, world):
    """The decode workload's description (both arms report the same one)."""
    bytes_layer, wbytes_layer = layer_bytes(synth.Q4_K)
    return {"workload": f"Llama-3.1-8B decode GEMV, batch 1: {nl} layers x "
                        "(q,k,v,o,gate,up,down), Q4_K weights, fp32 activations",
            "layers": nl,
            "weights_bytes_per_step": wbytes_layer * nl,
            "algorithmic_bytes_per_step": bytes_layer * nl,
            "l2": "working set 3.93 GB >> 129 MB L2: no flush between steps",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step decodes-then-dots a
    bounded sample (256 rows of each of the 7 matrices of one layer)."""
    import oracle
    cores = os.cpu_count() or 1
    rows = 256
    cache = {}

    def step(i):
        L = i % 4
        tot = 0
        for j, (name, N, K) in enumerate(SHAPES):
            key = (L, j)
            if key not in cache:
                w = synth.q4k_matrix(N, K, synth.layer_seed(SEED, L, j))
                cache[key] = (np.ascontiguousarray(w[:rows]),
                              synth.activations(1, K, synth.layer_seed(SEED + 1, L, j))[0])
            w, x = cache[key]
            oracle.gemv(synth.Q4_K, w, rows, K, x, nthreads=cores)
            tot += rows * synth.row_bytes(synth.Q4_K, K)
        return tot

    for i in range(min(args.warmup, 4)):
        step(i)
    for i in range(4):
        step(i)  # fill the input cache outside the timed region
    t0 = time.perf_counter()
    b = 0
    for i in range(args.steps):
        b += step(i)
    dt = time.perf_counter() - t0
    v = b / dt / 1e9
    sample = (f"per step: 256 rows of each of the 7 matrices of one Llama-3.1-8B layer "
              f"(Q4_K), fp64 decode-then-dot, OpenMP over rows on {cores} host threads")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(decode_config(args.layers, world),
                       timed_sample=f"{rows} rows x 7 matrices x 1 layer per step "
                                    "(layers cycled over 4 seeds); value = sampled "
                                    "algorithmic bytes / wall time"),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layers in the workload (32 = the full model; fewer only for profiling)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch directly instead of replaying a CUDA graph (profiling)")
    ap.add_argument("--only", choices=["prefill", "moe", "batched", "q8", "ffn", "tall"], default=None,
                    help="time just one secondary workload (profiling): the prefill GEMMs at "
                         "--prefill-m tokens, the OLMoE expert FFN, ..., or one decode GEMV on a "
                         "131072 x 4096 Q4_K matrix (the decode kernel's steady streaming rate)")
    ap.add_argument("--prefill-m", type=int, default=2048)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    if args.only:
        line = run_only(args, world, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    line = run_ours(args, world, rank, local)
    if rank == 0:
        line["cpu_baseline"] = time_oracle(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
