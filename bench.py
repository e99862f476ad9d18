#!/usr/bin/env python
"""Benchmark of the Q2_K weight-quantized matmul on GB300 (one JSON line).

Headline workload (``--workload decode_gemv_4096``): the decode GEMV
y = W x with M=1, N=K=4096 (5,505,024 bytes of Q2_K weights per matrix), x f32
~ N(0,1).  One step streams L distinct seeded weight matrices of that shape
(L chosen so they are at least 3x the L2 cache, so no weight byte is served
from L2) through one ``q2k_matmul`` launch each: L projections of one
activation x, each with its own W and y, so every call carries
Q2K_FLAG_INDEPENDENT (no call reads or writes what another writes) and
consecutive launches overlap.  The launches are captured once in a CUDA graph
and replayed.  ``secondary.decode_gemv_4096_dependent_chain`` times the same
matrices as a chain (each call's x is the previous call's y), where every
launch waits for the one before it.

``value``     weight bytes of all ranks / max-over-ranks step time (GB/s)
``roofline``  the dominant kernel (the GEMV): algorithmic bytes per launch
              (its weight bytes + x + y) / average launch time, against the
              measured HBM copy bandwidth
``e2e``       the same metric through the Python API, eager, with each step's
              activations copied in from pinned host memory and its outputs
              copied back inside the timed region (weights stay resident, as
              model weights do)
``secondary`` the other workloads: decode FFN pair, spec-verify M=16 with its
              embedding gather, prefill M=512 (TFLOP/s against the bf16 peak)
``cpu_baseline`` the CPU oracle (plain C, all host cores) on a bounded sample

``--impl reference`` times the CPU oracle alone on the same workload.
Under torchrun (N > 1) every rank runs an independent replica (weak scaling,
no collective on the data path); rank 0 prints.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import q2k_workloads as wl  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_gemv_4096")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dependent", action="store_true",
                    help="time the workload's matrices as dependent calls (each may read what "
                         "the one before wrote) instead of independent projections of one x")
    return ap.parse_args()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ggml_q2_quantized_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_key: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernels are unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None, None
    e = t.get(kernel_key, {}).get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None, None
    return e.get("dram_bytes_per_launch"), e.get("note")


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        # Let nvidia-smi finish starting up (its first query is slow) before the
        # timed region begins: wait for the first sample line.
        import select
        deadline = time.time() + 5.0
        self._first = ""
        while time.time() < deadline:
            r, _, _ = select.select([self.proc.stdout], [], [], 0.1)
            if r:
                self._first = self.proc.stdout.readline()
                break
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
            self.out = (getattr(self, "_first", "") or "") + (self.out or "")

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


# --------------------------------------------------------------------------- helpers

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def layers_for(weight_bytes: int, l2_bytes: int) -> int:
    return max(2, math.ceil(3 * l2_bytes / weight_bytes))


def batch_launches(m: int, n: int, k: int, layers: int, independent: bool) -> int:
    """Kernel launches of one q2k.MatmulBatch step of ``layers`` calls of one
    geometry on one x, as q2k_matmul_ex_batch enqueues them (with its scratch
    and per-geometry workspaces)."""
    if m <= 8:
        # fp32 GEMV, one launch per call; m = 1 calls on one x convert it once
        return layers + (1 if m == 1 and k // 64 <= 256 and layers >= 2 else 0)
    tiles = (n + 127) // 128
    if m <= 64:
        if independent and k % 1024 == 0 and layers >= 2 and tiles * layers >= 128:
            return 1 + -(-layers // 32)   # x image once, persistent grids of <= 32 calls
        return layers                     # small-m GEMM converts x itself
    splits = 1 if m > 128 or tiles >= 64 else 2
    if independent and splits == 1:
        return layers + 1                 # later calls reuse the first call's x image
    return 2 * layers                     # x image prepass + GEMM per call


def stack_of_weights(w: wl.Workload, layers: int, first: np.ndarray):
    """Layer 0 is the workload's own seeded matrix, layer l>0 draws from seed (w.seed, l)."""
    out = [first]
    nb = w.n * w.blocks_per_row
    for l in range(1, layers):
        out.append(wl.random_blocks(np.random.default_rng([w.seed, l]), nb))
    return out


def time_graph(torch, graph, stream, steps, warmup):
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps  # ms per step


def capture(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the path (one-time per-device setup happens here, not in capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def bench_matmul(torch, q2k, w: wl.Workload, steps, warmup, l2_bytes, device, with_e2e=False,
                 path="auto", independent=False, workspace="auto"):
    """Time a stack of distinct weight matrices of workload ``w`` (one launch each),
    all applied to the same x (independent projections when ``independent``)."""
    inp = wl.make_inputs(w, with_gather=False)
    layers = layers_for(w.weight_bytes, l2_bytes)
    ws = [torch.from_numpy(a).to(device) for a in stack_of_weights(w, layers, inp.w)]
    x = torch.from_numpy(inp.x).to(device)
    ys = torch.empty((layers, w.m, w.n), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)

    def step():
        for l in range(layers):
            q2k.matmul(x, ws[l], w.n, out=ys[l], path=path, independent=independent)

    batch_all = q2k.MatmulBatch([dict(x=x, w=ws[l], n=w.n, out=ys[l], path=path,
                                      independent=independent, workspace=workspace)
                                 for l in range(layers)])
    g = capture(torch, stream, batch_all.run)
    ms = time_graph(torch, g, stream, steps, warmup)
    res = {"layers": layers, "ms_per_step": ms, "us_per_call": ms * 1e3 / layers,
           "launches_per_step": layers}
    if with_e2e:
        x_host = torch.from_numpy(inp.x).pin_memory()
        y_host = torch.empty((layers, w.m, w.n), dtype=torch.float32).pin_memory()
        # the public batch API: the step's calls packed once and captured once
        # (q2k.MatmulBatch with graph=True), one graph launch per step
        batch = q2k.MatmulBatch([dict(x=x, w=ws[l], n=w.n, out=ys[l], path=path,
                                      independent=independent) for l in range(layers)],
                                graph=True)

        def timed(run_step):
            with torch.cuda.stream(stream):
                for _ in range(max(warmup, 3)):
                    x.copy_(x_host, non_blocking=True)
                    run_step()
                    y_host.copy_(ys, non_blocking=True)
                stream.synchronize()
                start = torch.cuda.Event(enable_timing=True)
                end = torch.cuda.Event(enable_timing=True)
                start.record(stream)
                for _ in range(steps):
                    x.copy_(x_host, non_blocking=True)
                    run_step()
                    y_host.copy_(ys, non_blocking=True)
                end.record(stream)
                end.synchronize()
            return start.elapsed_time(end) / steps

        res["e2e_ms_per_step"] = timed(batch.run)
        res["e2e_batch_ms_per_step"] = timed(batch_all.run)
        res["e2e_eager_ms_per_step"] = timed(step)
        res["h2d_bytes_per_step"] = x_host.numel() * 4
        res["d2h_bytes_per_step"] = y_host.numel() * 4
    return res


def bench_plain(torch, q2k, w: wl.Workload, steps, warmup, l2_bytes, device):
    """The stack of weight matrices through eager q2k.matmul calls without a
    workspace (the plain C call's path), timed with CUDA events on the stream."""
    inp = wl.make_inputs(w, with_gather=False)
    layers = layers_for(w.weight_bytes, l2_bytes)
    ws = [torch.from_numpy(a).to(device) for a in stack_of_weights(w, layers, inp.w)]
    x = torch.from_numpy(inp.x).to(device)
    ys = torch.empty((layers, w.m, w.n), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)

    def step():
        for l in range(layers):
            q2k.matmul(x, ws[l], w.n, out=ys[l], workspace=None)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        stream.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        end.synchronize()
    ms = start.elapsed_time(end) / steps
    return {"layers": layers, "ms_per_step": ms, "us_per_call": ms * 1e3 / layers}


def bench_chain(torch, q2k, w: wl.Workload, steps, warmup, l2_bytes, device):
    """The stack as a dependent chain (N = K): x of call l + 1 is y of call l."""
    assert w.m == 1 and w.n == w.k
    inp = wl.make_inputs(w, with_gather=False)
    layers = layers_for(w.weight_bytes, l2_bytes)
    ws = [torch.from_numpy(a).to(device) for a in stack_of_weights(w, layers, inp.w)]
    acts = torch.empty((layers + 1, 1, w.k), dtype=torch.float32, device=device)
    acts[0].copy_(torch.from_numpy(inp.x))
    stream = torch.cuda.Stream(device)

    def step():
        for l in range(layers):
            q2k.matmul(acts[l], ws[l], w.n, out=acts[l + 1], const_weights=True)

    g = capture(torch, stream, step)
    ms = time_graph(torch, g, stream, steps, warmup)
    us = ms * 1e3 / layers
    return {"us_per_call": us, "weight_GBps": w.weight_bytes / (us * 1e-6) / 1e9,
            "m": 1, "n": w.n, "k": w.k, "path": "gemv", "matrices_per_step": layers,
            "calls": "each call's x is the previous call's y (Q2K_FLAG_CONST_WEIGHTS)"}


def bench_batched(torch, q2k, w: wl.Workload, batches, steps, warmup, l2_bytes, device):
    """``batches`` GEMVs of workload ``w`` per batched launch, a stack of distinct
    batched weight buffers (larger than L2 together), one launch each."""
    assert w.m == 1
    per = w.weight_bytes
    layers = layers_for(per * batches, l2_bytes)
    inp = wl.make_inputs(w, with_gather=False)
    mats = stack_of_weights(w, batches, inp.w)  # `batches` distinct matrices
    bufs = []
    for l in range(layers):
        # rotate the matrices so every buffer differs in order (distinct addresses anyway)
        bufs.append(torch.from_numpy(np.concatenate(mats[l % batches:] + mats[:l % batches]))
                    .to(device))
    x = torch.from_numpy(wl.random_activations(np.random.default_rng([w.seed, 99]), batches,
                                               w.k)).to(device)
    ys = torch.empty((layers, batches, w.n), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)

    def step():
        for l in range(layers):
            q2k.matmul_batched_mv(x, bufs[l], w.n, out=ys[l])

    g = capture(torch, stream, step)
    ms = time_graph(torch, g, stream, steps, warmup)
    us = ms * 1e3 / layers
    return {"us_per_launch": us, "weight_GBps": batches * per / (us * 1e-6) / 1e9,
            "batches": batches, "n": w.n, "k": w.k, "launches_per_step": layers,
            "path": "gemv (batched, one launch)"}


def bench_routed(torch, q2k, rw, steps, warmup, device):
    """mm_id over a pool of ``rw.n_experts`` experts; each launch of a step uses
    its own ids (fresh experts), so weights come from HBM, not L2."""
    rng = np.random.default_rng(rw.seed)
    distinct = 4  # distinct expert matrices, tiled over the pool (timing only)
    base = [wl.random_blocks(rng, rw.n * (rw.k // wl.QK_K)) for _ in range(distinct)]
    pool = torch.from_numpy(np.concatenate([base[e % distinct] for e in range(rw.n_experts)])
                            ).to(device)
    x = torch.from_numpy(wl.random_activations(rng, rw.n_tokens, rw.k)).to(device)
    launches = 16
    ids = [torch.from_numpy(wl.make_routed_ids(rw, i).view(np.int32)).to(device)
           for i in range(launches)]
    routes = rw.n_tokens * rw.top_k
    ys = torch.empty((launches, routes, rw.n), dtype=torch.float32, device=device)
    bad = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device)

    def step():
        for i in range(launches):
            q2k.matmul_id(x, pool, ids[i], rw.n, rw.n_experts, rw.top_k, out=ys[i], check=False)

    g = capture(torch, stream, step)
    ms = time_graph(torch, g, stream, steps, warmup)
    us = ms * 1e3 / launches
    uniq = np.mean([len(set(wl.make_routed_ids(rw, i).tolist())) for i in range(launches)])
    return {"us_per_launch": us, "weight_GBps": uniq * rw.expert_bytes / (us * 1e-6) / 1e9,
            "n_tokens": rw.n_tokens, "top_k": rw.top_k, "n": rw.n, "k": rw.k,
            "n_experts": rw.n_experts, "expert_bytes": rw.expert_bytes,
            "unique_experts_per_launch": float(uniq), "path": "gemv per route (one launch)"}


def bench_routed_tc(torch, q2k, rw, steps, warmup, device, peaks):
    """mm_id on the tensor path (routes grouped per expert, bf16 MMAs): one
    launch sequence (routing, x gather, GEMM) per step, fresh ids each step."""
    rng = np.random.default_rng(rw.seed)
    pool = torch.from_numpy(np.concatenate([wl.random_blocks(rng, rw.n * (rw.k // wl.QK_K))
                                            for _ in range(rw.n_experts)])).to(device)
    x = torch.from_numpy(wl.random_activations(rng, rw.n_tokens, rw.k)).to(device)
    launches = 4
    ids = [torch.from_numpy(wl.make_routed_ids(rw, i).view(np.int32)).to(device)
           for i in range(launches)]
    routes = rw.n_tokens * rw.top_k
    ys = torch.empty((launches, routes, rw.n), dtype=torch.float32, device=device)
    ws = torch.empty(q2k.matmul_id_workspace_bytes(rw.n_tokens, rw.top_k, rw.n, rw.k,
                                                   rw.n_experts, path="tensor"),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)

    def step():
        for i in range(launches):
            q2k.matmul_id_ex(x, pool, ids[i], rw.n, rw.n_experts, rw.top_k, path="tensor",
                             out=ys[i], check=False, workspace=ws)

    g = capture(torch, stream, step)
    ms = time_graph(torch, g, stream, steps, warmup)
    us = ms * 1e3 / launches
    tflops = 2.0 * routes * rw.n * rw.k / (us * 1e-6) / 1e12
    return {"us_per_launch": us, "TFLOPs": tflops,
            "frac_bf16_measured": tflops / peaks["bf16_tflops"],
            "weight_GBps": rw.n_experts * rw.expert_bytes / (us * 1e-6) / 1e9,
            "n_tokens": rw.n_tokens, "top_k": rw.top_k, "n": rw.n, "k": rw.k,
            "n_experts": rw.n_experts, "path": "tensor (routes tiled per expert)"}


def bench_gather(torch, q2k, w: wl.Workload, steps, warmup, device):
    inp = wl.make_inputs(w)
    table = torch.from_numpy(inp.table).to(device)
    ids = torch.from_numpy(inp.ids.astype(np.int32)).to(device)
    out = torch.empty((w.gather_tokens, w.k), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    reps = 64

    def step():
        for _ in range(reps):
            q2k.embedding_gather(table, ids, w.k, out=out, check=False)

    g = capture(torch, stream, step)
    ms = time_graph(torch, g, stream, steps, warmup)
    return {"us_per_call": ms * 1e3 / reps, "n_tokens": w.gather_tokens,
            "table": f"{w.gather_vocab}x{w.k}"}


def cpu_baseline(w: wl.Workload, budget_s: float = 12.0):
    import oracle
    inp = wl.make_inputs(w, with_gather=False)
    cores = os.cpu_count() or 1
    # bounded sample: whole weight rows of the workload, all x rows
    rows = w.n
    if w.m * w.n * w.k > 2e9:
        rows = max(1, int(2e9 // (w.m * w.k)))
    row_bytes = w.blocks_per_row * wl.BLOCK_BYTES
    wsub = inp.w[: rows * row_bytes]
    oracle.matmul(inp.x, wsub, rows, threads=cores)  # warm (build + page-in)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.matmul(inp.x, wsub, rows, threads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s or reps >= 100000:
            break
    sec = el / reps
    return {"value": rows * row_bytes / sec / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x oracle matmul of {w.name} (M={w.m}, {rows} of {w.n} weight rows,"
                      f" K={w.k}), {cores} threads, {el:.1f} s",
            "flops_per_s": 2 * w.m * rows * w.k / sec}


# --------------------------------------------------------------------------- arms

def headline_parity(w: wl.Workload, inp, y) -> dict:
    """The headline launch's y (layer 0: the workload's seeded matrix and x)
    against the oracle, |y - y_ref| / S per output (part of the CPU-baseline
    leg, the one place besides the tests that runs the oracle)."""
    import oracle
    yref, s = oracle.matmul(inp.x, inp.w, w.n, threads=os.cpu_count() or 1)
    err = np.abs(y.astype(np.float64) - yref)
    tol = 1e-5 if w.m <= 8 else 8e-3
    ratio = np.where(s > 0, err / np.maximum(s, 1e-300), 0.0)
    return {"max_err_over_S": float(ratio.max()), "tolerance_over_S": tol,
            "within_tolerance": bool((err <= tol * s).all()),
            "outputs": int(y.size), "reference": "CPU oracle (f64 sum of the page's f32 weights)"}


def run_reference(args):
    world, rank, _ = dist_setup()
    w = wl.by_name(args.workload)
    if rank != 0:
        return 0
    import oracle
    inp = wl.make_inputs(w, with_gather=False)
    cores = os.cpu_count() or 1
    rows = w.n if w.m * w.n * w.k <= 2e9 else max(1, int(2e9 // (w.m * w.k)))
    row_bytes = w.blocks_per_row * wl.BLOCK_BYTES
    wsub = inp.w[: rows * row_bytes]
    for _ in range(args.warmup):
        oracle.matmul(inp.x, wsub, rows, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(inp.x, wsub, rows, threads=cores)
    el = time.perf_counter() - t0
    value = args.steps * rows * row_bytes / el / 1e9
    sample = (f"each step: oracle matmul of {w.name} (M={w.m}, {rows} of {w.n} weight rows,"
              f" K={w.k}) on {cores} host threads")
    line = {"impl": "reference", "metric": "q2k_matmul_weight_GBps", "value": value,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from ggml_q2_quantized_gb300 import build as lib_build
    import ggml_q2_quantized_gb300 as q2k
    lib_build.build()
    q2k.load()

    peaks, peak_kind = load_peaks()
    props = torch.cuda.get_device_properties(device)
    l2_bytes = getattr(props, "L2_cache_size", 0) or 126 * 2**20
    w = wl.by_name(args.workload)
    steps, warmup = args.steps, max(3, args.warmup)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- headline: the timed region
    inp = wl.make_inputs(w, with_gather=False)
    layers = layers_for(w.weight_bytes, l2_bytes)
    ws = [torch.from_numpy(a).to(device) for a in stack_of_weights(w, layers, inp.w)]
    x = torch.from_numpy(inp.x).to(device)
    ys = torch.empty((layers, w.m, w.n), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)

    indep = not args.dependent
    # the step's calls packed once: q2k_matmul_ex_batch enqueues them; as
    # independent projections of this x, x is converted once into the batch's
    # scratch (m = 1: the GEMV's form; m <= 64: the bf16 image that persistent
    # tensor grids share; m > 64: the workspace image later calls reuse)
    batch = q2k.MatmulBatch([dict(x=x, w=ws[l], n=w.n, out=ys[l], independent=indep)
                             for l in range(layers)])
    launches_per_step = batch_launches(w.m, w.n, w.k, layers, indep)

    def step():
        batch.run()

    graph = capture(torch, stream, step)
    for _ in range(warmup):
        graph.replay()
    barrier()
    # The timed region: `steps` steps, timed with CUDA events on the replay
    # stream, repeated back to back until the repeats cover >= 1 s (so the
    # clock sampler sees the load); the median repeat is reported.
    probe_s = torch.cuda.Event(enable_timing=True)
    probe_e = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        probe_s.record(stream)
        for _ in range(steps):
            graph.replay()
        probe_e.record(stream)
    probe_e.synchronize()
    repeats = max(1, min(2000, math.ceil(1000.0 / max(probe_s.elapsed_time(probe_e), 1e-3))))
    if world > 1:
        t = torch.tensor([repeats], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        repeats = int(t.item())
    barrier()
    with ClockSampler(device.index) as clk:
        barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(repeats)]
        with torch.cuda.stream(stream):
            for start, end in evs:
                start.record(stream)
                for _ in range(steps):
                    graph.replay()
                end.record(stream)
        evs[-1][1].synchronize()
        barrier()
    per_repeat = [a.elapsed_time(b) / steps for a, b in evs]
    ms = statistics.median(per_repeat)
    if world > 1:
        t = torch.tensor([ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    y_check = ys[0].cpu().numpy()   # layer 0: the workload's own matrix and x
    assert q2k.device_error() == 0
    bytes_per_step = layers * w.weight_bytes
    value = world * bytes_per_step / (ms * 1e-3) / 1e9
    launch_us = ms * 1e3 / layers
    algo_bytes = w.weight_bytes + 4 * w.m * w.k + 4 * w.m * w.n
    achieved = algo_bytes / (launch_us * 1e-6) / 1e9
    kernel_key = "gemv" if w.m <= 8 else "tensor"
    traffic, traffic_note = traffic_for(kernel_key, w.name)

    line = {
        "metric": "q2k_matmul_weight_GBps",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.m <= 8 else "bf16", "data": "synthetic",
        "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k,
                   "weight_bytes_per_matrix": w.weight_bytes, "matrices_per_step": layers,
                   "l2_policy": f"inputs larger than L2: {layers} distinct weight matrices "
                                f"({bytes_per_step / 2**20:.0f} MiB) per step vs "
                                f"{l2_bytes / 2**20:.0f} MiB L2",
                   "timing": (f"CUDA graph of the step's launches, CUDA events on the replay "
                              f"stream; {repeats} back-to-back repeats of the {steps} timed steps, "
                              f"median repeat reported (spread {min(per_repeat):.4f}-"
                              f"{max(per_repeat):.4f} ms per step)"),
                   "calls": ("independent projections of one x (Q2K_FLAG_INDEPENDENT) enqueued as "
                             "one q2k.MatmulBatch: x converted once per step" if indep
                             else "dependent calls, one launch per matrix, as one q2k.MatmulBatch"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_call": launch_us,
        "gpu_launches": steps * launches_per_step,
        "roofline": {"bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": algo_bytes,
                     "kernel": "q2k gemv_m1_kernel" if w.m == 1 else f"q2k {kernel_key}",
                     "frac_of_nominal_8TBps": achieved / 8000.0},
    }
    if w.m <= 8:
        # The exact fp32 GEMV is bound by arithmetic issue, not by HBM: every
        # weight takes one 2-cycle integer mask and two fp32 FMAs (the weight
        # and the dot, 1 cycle each per 32 lanes), i.e. 4 sub-partition cycles
        # per 32 weights on each of the 4 sub-partitions of the SMs.  Its peak
        # in weight bytes per second at the SM clock of the run:
        props = torch.cuda.get_device_properties(device)
        sm_mhz = clk.summary().get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
        weights_per_s = props.multi_processor_count * 4 * (32 / 4) * sm_mhz * 1e6
        alu_peak = weights_per_s * wl.BLOCK_BYTES / 256 / 1e9
        hbm = dict(line["roofline"])
        line["roofline"] = {
            "bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "GB/s",
            "frac": achieved / alu_peak, "traffic": traffic,
            "peak_source": (f"issue bound of the exact fp32 decode + dot (1 integer mask at 2 cycles "
                            f"and 2 fp32 FMAs at 1 cycle per 32 weights per sub-partition), "
                            f"{props.multi_processor_count} SMs x 4 sub-partitions at the run's "
                            f"median SM clock {sm_mhz:.0f} MHz"),
            "algorithmic_bytes_per_launch": algo_bytes,
            "kernel": hbm["kernel"],
            "hbm": {"peak": hbm["peak"], "frac": hbm["frac"], "peak_source": hbm["peak_source"],
                    "frac_of_nominal_8TBps": hbm["frac_of_nominal_8TBps"]}}
    if traffic_note:
        line["roofline"]["traffic_note"] = traffic_note
    line["clocks"] = clk.summary()

    # ---- e2e through the public API (eager), host buffers, copies inside the region
    e2e = bench_matmul(torch, q2k, w, steps, warmup, l2_bytes, device, with_e2e=True,
                       independent=indep)
    line["e2e"] = {"value": world * bytes_per_step / (e2e["e2e_ms_per_step"] * 1e-3) / 1e9,
                   "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                   "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                   "ms_per_step": e2e["e2e_ms_per_step"],
                   "how": "the public batch API: the step's calls (one per weight matrix, as "
                          "the headline) packed once in a q2k.MatmulBatch(graph=True), whose first "
                          "run captures its q2k_matmul_ex_batch call in a CUDA graph (one graph "
                          "launch per step after that), with the activations copied from pinned "
                          "host memory and all outputs copied back each step",
                   "batch_value": world * bytes_per_step / (e2e["e2e_batch_ms_per_step"] * 1e-3) / 1e9,
                   "batch_how": "the same with q2k.MatmulBatch(graph=False): one "
                                "q2k_matmul_ex_batch call enqueues every launch each step",
                   "eager_value": world * bytes_per_step / (e2e["e2e_eager_ms_per_step"] * 1e-3) / 1e9,
                   "eager_how": "the same step as one eager q2k.matmul call per weight matrix"}

    # ---- secondary workloads (not the headline; reported for the metric's M=512 half)
    if not args.no_secondary:
        sec = {}
        for name in ("ffn_pair", "ffn_pair_down", "spec_verify_m16", "prefill_m512"):
            sw = wl.by_name(name)
            # the step's calls are projections of one x, each with its own W
            # and y (Q2K_FLAG_INDEPENDENT: the GEMV and the small-m tensor
            # path fetch their inputs before the dependency wait; at M = 512
            # the batch converts x once and the GEMMs overlap)
            r = bench_matmul(torch, q2k, sw, max(3, steps // 4), 3, l2_bytes, device,
                             independent=True)
            us = r["us_per_call"]
            entry = {"us_per_call": us, "weight_GBps": sw.weight_bytes / (us * 1e-6) / 1e9,
                     "TFLOPs": sw.flops / (us * 1e-6) / 1e12, "m": sw.m, "n": sw.n, "k": sw.k,
                     "path": "gemv" if sw.m <= 8 else "tensor", "matrices_per_step": r["layers"]}
            entry["frac_hbm_measured"] = entry["weight_GBps"] / peaks["hbm_gbs"]
            if sw.m > 8:
                entry["frac_bf16_measured"] = entry["TFLOPs"] / peaks["bf16_tflops"]
                entry["frac_bf16_nominal_2250"] = entry["TFLOPs"] / 2250.0
            sec[name] = entry
        # the M=512 workload through the plain call without a workspace (as a C
        # caller of q2k_matmul makes it: eager launches, the library's own
        # scratch for the x image; a graph capture would take the in-kernel
        # conversion instead)
        sw = wl.by_name("prefill_m512")
        r = bench_plain(torch, q2k, sw, max(3, steps // 4), 3, l2_bytes, device)
        us = r["us_per_call"]
        sec["prefill_m512_plain_c_call"] = {
            "us_per_call": us, "TFLOPs": sw.flops / (us * 1e-6) / 1e12,
            "frac_bf16_measured": sw.flops / (us * 1e-6) / 1e12 / peaks["bf16_tflops"],
            "m": sw.m, "n": sw.n, "k": sw.k, "path": "tensor, no workspace (q2k_matmul)",
            "matrices_per_step": r["layers"]}
        # the M=16 workload through the fp32 GEMV path as well (forced)
        sw = wl.by_name("spec_verify_m16")
        r = bench_matmul(torch, q2k, sw, max(3, steps // 4), 3, l2_bytes, device, path="gemv")
        us = r["us_per_call"]
        sec["spec_verify_m16_gemv_path"] = {
            "us_per_call": us, "weight_GBps": sw.weight_bytes / (us * 1e-6) / 1e9,
            "TFLOPs": sw.flops / (us * 1e-6) / 1e12, "m": sw.m, "n": sw.n, "k": sw.k,
            "path": "gemv", "matrices_per_step": r["layers"]}
        if w.m == 1 and w.n == w.k:
            sec[f"{w.name}_dependent_chain"] = bench_chain(torch, q2k, w, max(3, steps // 4), 3,
                                                           l2_bytes, device)
        sec["spec_verify_gather"] = bench_gather(torch, q2k, wl.by_name("spec_verify_m16"),
                                                 max(3, steps // 4), 3, device)
        bb = wl.BATCHED_DECODE_BATCHES
        r = bench_batched(torch, q2k, wl.by_name("decode_gemv_4096"), bb, max(3, steps // 4), 3,
                          l2_bytes, device)
        r["frac_hbm_measured"] = r["weight_GBps"] / peaks["hbm_gbs"]
        sec[f"batched_mv_{bb}x4096"] = r
        r = bench_routed(torch, q2k, wl.MOE_DECODE, max(3, steps // 4), 3, device)
        r["frac_hbm_measured"] = r["weight_GBps"] / peaks["hbm_gbs"]
        sec[wl.MOE_DECODE.name] = r
        sec[wl.MOE_PREFILL.name] = bench_routed_tc(torch, q2k, wl.MOE_PREFILL, max(3, steps // 4),
                                                   3, device, peaks)
        line["secondary"] = sec
        assert q2k.device_error() == 0

    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
        line["parity"] = headline_parity(w, inp, y_check)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
