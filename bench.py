"""Benchmark of the NVFP4 linear layer on GB300.

One step is one decode pass of the 27B-class workload at M = 1: the up and
gate projections (5120 -> 17408), the down projection (17408 -> 5120) and the
LM head (5120 -> 151936), each Y = X W^T with an NVFP4 weight resident in
HBM.  The metric is the rate at which the step streams its algorithmic bytes
(NVFP4 weight bytes + bf16 X and Y), in GB/s, next to the HBM roofline.  The
weights of one step (588 MB) exceed the 129 MB L2, so every step reads them
from HBM.

Also reported (same JSON line): the prefill GEMM on the block-scaled FP4
tensor-core path when the library provides it, the per-M skinny decode
rates, and the quantizer.

The CPU baseline is the oracle (plain single-threaded C++, fp64 matmul) timed
on a bounded row sample of the same workload.  ``--impl reference`` times only
that oracle, as the reference arm.
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

import synth  # noqa: E402

WORKLOAD = "decode_27b"
METRIC = "NVFP4 GEMV HBM GB/s (% of GB300 peak) at M=1; prefill FP4 TFLOPS (% peak)"


def step_bytes(lins) -> int:
    """Algorithmic bytes of one decode step: NVFP4 weights + bf16 X + bf16 Y."""
    return sum(l.weight_bytes + 2 * l.M * l.K + 2 * l.M * l.N for l in lins)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        self.t_start = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)  # let the sampler start before the timed region
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(lins, budget_s: float, max_rows: int | None = None):
    """Time the oracle's decode GEMV (dequant + fp64 matmul) on leading rows of
    each weight of the workload.  Returns (GB/s of NVFP4 weight, seconds,
    description).  Quantization of the sampled rows happens before the clock."""
    import oracle

    prepared = []
    for l in lins:
        rows = max_rows or max(8, min(l.N, 512))
        wb = l.weight_bf16(0, rows)
        _, ts, _ = oracle.tensor_scale(wb)
        c, s = oracle.quantize_rows(wb, ts)
        prepared.append((l, c, s, ts, l.act_bf16(), rows))
    done_bytes, t0, calls = 0, time.perf_counter(), 0
    while True:
        for l, c, s, ts, x, rows in prepared:
            oracle.reference_gemm(x, l.M, c, s, ts)
            done_bytes += rows * (l.K // 2 + l.K // 16)
            calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    desc = (f"oracle decode GEMV (dequant + fp64 matmul, 1 thread) on the first "
            f"{prepared[0][5]} rows of each of {len(lins)} weights, {calls} calls")
    return done_bytes / dt / 1e9, dt, desc


def _oracle_slice_worker(job):
    """One process of the all-core CPU baseline: the oracle's decode GEMV on
    its own block of rows of each weight, repeated for `budget_s` seconds.
    Returns (bytes of NVFP4 weight processed, seconds)."""
    name, part, rows, budget_s = job
    import oracle

    prepared = []
    for l in synth.workload(name):
        r0 = min(part * rows, max(0, l.N - rows))
        wb = l.weight_bf16(r0, rows)
        _, ts, _ = oracle.tensor_scale(wb)
        c, s = oracle.quantize_rows(wb, ts)
        prepared.append((l, c, s, ts, l.act_bf16()))
    done, t0 = 0, time.perf_counter()
    while True:
        for l, c, s, ts, x in prepared:
            oracle.reference_gemm(x, l.M, c, s, ts)
            done += rows * (l.K // 2 + l.K // 16)
        if time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0


def cpu_oracle_all_cores(workload: str, budget_s: float, rows: int = 256):
    """The oracle as N independent copies, one process per core of this
    process's affinity mask, each on its own row block (spawned processes:
    nothing forked after the GPU was touched).  Returns (GB/s, cores, desc)."""
    import multiprocessing as mp

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_slice_worker, [(workload, i, rows, budget_s) for i in range(cores)])
    gbs = sum(b / t for b, t in res) / 1e9
    desc = (f"oracle decode GEMV (dequant + fp64 matmul), {cores} processes, each on its own "
            f"{rows}-row block of every weight of {workload} for ~{budget_s:.0f} s")
    return gbs, cores, desc


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time; every rank gets it (no-op on one process)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    lins = synth.workload(args.workload)
    per_step = []
    for _ in range(args.warmup):
        cpu_oracle_sample(lins, 0.0, max_rows=64)
    gbs_all = []
    for _ in range(args.steps):
        gbs, dt, desc = cpu_oracle_sample(lins, 0.0, max_rows=256)
        per_step.append(dt)
        gbs_all.append(gbs)
    gbs = statistics.median(gbs_all)
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(per_step), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "M": 1, "shapes_KxN": [[l.K, l.N] for l in lins],
                       "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def run_native(args):
    import torch
    import torch.distributed as dist

    import nvfp4_weight_quantized_02_gb300 as pkg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.load()

    # ---- inputs resident in HBM (weights quantized on device; not timed)
    lins = synth.workload(args.workload)
    weights, xs, ys = [], [], []
    for l in lins:
        wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        weights.append(pkg.quantize(wb))
        del wb
        xs.append(torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev))
        ys.append(torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev))
    # X and Y of all problems as views into one buffer each, so a step's
    # inputs arrive with one host-to-device copy and its results leave with
    # one device-to-host copy (offsets stay 16-byte aligned: K, N % 8 == 0)
    xcat = torch.empty(sum(x.numel() for x in xs), dtype=torch.bfloat16, device=dev)
    ycat = torch.empty(sum(y.numel() for y in ys), dtype=torch.bfloat16, device=dev)
    ox = oy = 0
    for i, l in enumerate(lins):
        v = xcat[ox:ox + l.M * l.K].view(l.M, l.K)
        v.copy_(xs[i])
        xs[i] = v
        ys[i] = ycat[oy:oy + l.M * l.N].view(l.M, l.N)
        ox += l.M * l.K
        oy += l.M * l.N
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # one workspace per problem, allocated once (the FP4 decode path's split X,
    # partial sums and counters)
    wss = [torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K), 16),
                       dtype=torch.uint8, device=dev) for l in lins]
    plans = [pkg.imp_nvfp4_gemm_plan(l.M, l.N, l.K) for l in lins]
    torch.cuda.synchronize()

    def step():
        for x, w, y, ws in zip(xs, weights, ys, wss):
            pkg.gemm(x, w, y=y, dev_status=status, stream=stream, workspace=ws)

    # per-kernel timing events (on the launching stream)
    def timed_steps(k, per_kernel):
        evs = []
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(k):
            if per_kernel:
                row = []
                for x, w, y, ws in zip(xs, weights, ys, wss):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    pkg.gemm(x, w, y=y, dev_status=status, stream=stream, workspace=ws)
                    e1.record(stream)
                    row.append((e0, e1))
                evs.append(row)
            else:
                step()
        end.record(stream)
        return start, end, evs

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        start, end, _ = timed_steps(args.steps, per_kernel=False)
        torch.cuda.synchronize()
        elapsed_ms = start.elapsed_time(end)
        # second pass with per-kernel events (for the roofline of the top kernel)
        _, _, evs = timed_steps(args.steps, per_kernel=True)
        torch.cuda.synchronize()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    if world > 1:
        dist.barrier()
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")

    per_kernel_ms = [statistics.mean(row[i][0].elapsed_time(row[i][1]) for row in evs)
                     for i in range(len(lins))]
    bytes_step = step_bytes(lins)
    ms_per_step = elapsed_ms / args.steps
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9

    # ---- e2e through the public API with host buffers
    pin_x = torch.empty(xcat.shape, dtype=torch.bfloat16, pin_memory=True).copy_(xcat)
    pin_y = torch.empty(ycat.shape, dtype=torch.bfloat16, pin_memory=True)
    h2d = pin_x.numel() * 2
    d2h = pin_y.numel() * 2

    def e2e_step():
        xcat.copy_(pin_x, non_blocking=True)
        for x, w, y, ws in zip(xs, weights, ys, wss):
            pkg.gemm(x, w, y=y, dev_status=status, stream=stream, workspace=ws)
        pin_y.copy_(ycat, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    e2e_value = world * bytes_step / (e2e_ms * 1e-3) / 1e9

    hbm_peak, _, peak_kind = load_peaks()
    top = int(np.argmax(per_kernel_ms))
    top_bytes = lins[top].weight_bytes + 2 * lins[top].K + 2 * lins[top].N
    achieved = top_bytes / (per_kernel_ms[top] * 1e-3) / 1e9
    top_kernel = plans[top][1]
    traffic = load_traffic(top_kernel, lins[top])
    # The same kernel launched back to back (its weight alone exceeds L2, so
    # every launch reads it from HBM): the launch interval once start-up
    # overlaps the previous launch, next to the isolated duration above.
    xt, wt, yt, wst = xs[top], weights[top], ys[top], wss[top]
    for _ in range(3):
        pkg.gemm(xt, wt, y=yt, dev_status=status, stream=stream, workspace=wst)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    reps = 20
    e0.record(stream)
    for _ in range(reps):
        pkg.gemm(xt, wt, y=yt, dev_status=status, stream=stream, workspace=wst)
    e1.record(stream)
    torch.cuda.synchronize()
    b2b_ms = e0.elapsed_time(e1) / reps
    b2b_gbs = top_bytes / (b2b_ms * 1e-3) / 1e9

    extra = {}
    if rank == 0 and not args.no_extra:
        extra = bench_extras(args, pkg, dev, stream, hbm_peak)
        # the same step replayed as one CUDA graph (the decode launches of a
        # step captured once; programmatic dependent launch edges kept)
        try:
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                for x, w, y, ws in zip(xs, weights, ys, wss):
                    pkg.gemm(x, w, y=y, dev_status=status, stream=cap, workspace=ws)
            torch.cuda.synchronize()
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            gstream = torch.cuda.current_stream(dev)
            g0.record(gstream)
            for _ in range(args.steps):
                graph.replay()
            g1.record(gstream)
            torch.cuda.synchronize()
            gms = g0.elapsed_time(g1) / args.steps
            if int(status.item()) != 0:
                raise RuntimeError(f"device status {int(status.item())} in the graph replay")
            extra["decode_graph_replay"] = {
                "ms_per_step": gms, "GB/s": bytes_step / (gms * 1e-3) / 1e9,
                "frac_of_hbm_peak": bytes_step / (gms * 1e-3) / 1e9 / hbm_peak}
            del graph
        except Exception as e:  # report, do not fail the benchmark line
            extra["decode_graph_replay"] = {"error": str(e)[:200]}
        # the same step on weights prepared once in the MMA layout (contiguous
        # 16 KB code tiles, scale atoms) through imp_nvfp4_gemm_mma
        prepared = [pkg.prepare_mma(w, stream=stream) for w in weights]
        pws = [torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K), 16),
                           dtype=torch.uint8, device=dev) for l in lins]

        def prepared_step():
            for x, w, y, ws in zip(xs, prepared, ys, pws):
                pkg.gemm_mma(x, w, y=y, dev_status=status, stream=stream, workspace=ws)

        for _ in range(args.warmup):
            prepared_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            prepared_step()
        e1.record(stream)
        torch.cuda.synchronize()
        pms = e0.elapsed_time(e1) / args.steps
        extra["decode_prepared_mma_layout"] = {
            "ms_per_step": pms, "GB/s": bytes_step / (pms * 1e-3) / 1e9,
            "frac_of_hbm_peak": bytes_step / (pms * 1e-3) / 1e9 / hbm_peak}
        del prepared, pws
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the prepared step")

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 weights, bf16 x/y, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": 1, "shapes_KxN": [[l.K, l.N] for l in lins],
                   "bytes_per_step": bytes_step, "l2": "inputs larger than L2 (588 MB per step)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm_peak": value / world / hbm_peak,
        "per_kernel_us": {l.name: 1e3 * t for l, t in zip(lins, per_kernel_ms)},
        "per_kernel_gbs": {l.name: (l.weight_bytes + 2 * l.K + 2 * l.N) / (t * 1e-3) / 1e9
                           for l, t in zip(lins, per_kernel_ms)},
        "roofline": {"bound": "hbm", "kernel": f"{top_kernel} ({lins[top].name} "
                     f"{lins[top].K}x{lins[top].N})", "achieved": achieved, "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": traffic,
                     "back_to_back": {"us_per_launch": 1e3 * b2b_ms, "achieved": b2b_gbs,
                                      "frac": b2b_gbs / hbm_peak}},
        "gpu_launches": args.steps * sum(n for n, _ in plans),
        "kernels": {l.name: {"kernel": k, "launches_per_call": n} for l, (n, k) in zip(lins, plans)},
        "clocks": clocks.summary(),
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu_baseline:
        gbs, dt, desc = cpu_oracle_sample(lins, args.cpu_seconds)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": dt}
        if world == 1:
            try:
                gbs, cores, desc = cpu_oracle_all_cores(args.workload, args.cpu_seconds)
                line["cpu_baseline_all_cores"] = {"value": gbs, "unit": "GB/s", "cores": cores,
                                                  "kind": "oracle", "sample": desc}
            except Exception as e:  # report, do not lose the benchmark line
                line["cpu_baseline_all_cores"] = {"error": str(e)[:200]}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def load_traffic(kernel: str, lin):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries
    (profiles/traffic.json), if one is recorded for this shape."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        return t.get(f"{kernel}:{lin.K}x{lin.N}")
    except (OSError, ValueError):
        return None


def fp4_peak_tflops():
    """Dense FP4 tensor peak: the measured bf16 peak times the nominal
    FP4 : bf16 ratio (13.5 : 2.25 PFLOP/s dense)."""
    _, bf16, kind = load_peaks()
    return bf16 * (13.5 / 2.25), kind


def bench_prefill(args, pkg, dev, stream):
    """Prefill GEMMs (M = 2048): the block-scaled FP4 tensor-core GEMM alone
    (X already quantized, W scales in the atom layout) and the whole
    imp_nvfp4_gemm call (X quantization + W scale layout + GEMM)."""
    import torch

    peak, kind = fp4_peak_tflops()
    res = {}
    for l in synth.workload("prefill_27b"):
        wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        w = pkg.quantize(wb)
        del wb
        wm = pkg.prepare_mma(w)
        x = torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        xq = pkg.quantize_mma(x)
        y = torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K), dtype=torch.uint8,
                         device=dev)
        wsf = torch.empty(pkg.imp_nvfp4_gemm_fp4_workspace_size(l.M, l.N, l.K),
                          dtype=torch.uint8, device=dev)
        flops = 2.0 * l.M * l.N * l.K
        out = {}
        for name, fn in (("gemm_fp4", lambda: pkg.gemm_fp4(xq, wm, y=y, stream=stream)),
                         ("gemm_fp4_stream_k", lambda: pkg.gemm_fp4(xq, wm, y=y, stream=stream,
                                                                    workspace=wsf,
                                                                    stream_k=True)),
                         ("imp_nvfp4_gemm", lambda: pkg.gemm(x, w, y=y, stream=stream,
                                                             workspace=ws))):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            reps = 20
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / reps
            tf = flops / (t * 1e-3) / 1e12
            out[name] = {"us": 1e3 * t, "TFLOP/s": tf, "frac_of_fp4_peak": tf / peak}
        res[f"M{l.M}_{l.K}x{l.N}"] = out
        del w, wm, x, xq, y, ws
    res["fp4_peak_tflops"] = peak
    res["fp4_peak_kind"] = f"{kind} bf16 x 6 (nominal fp4:bf16 ratio)"
    return res


def bench_extras(args, pkg, dev, stream, hbm_peak):
    """Prefill GEMMs, skinny-M decode rates (M = 2..16) and the quantizer rate."""
    import torch

    out = {"prefill": bench_prefill(args, pkg, dev, stream)}
    # Skinny M: back-to-back calls cycling through copies of W whose total
    # exceeds L2 twice over, so each call reads its weight from HBM (no flush
    # kernel between calls, which would idle the GPU and hide start-up cost).
    lins = synth.workload("skinny_27b")
    skinny = {}
    cache = {}
    l2 = 129 * 1024 * 1024
    for l in lins:
        key = (l.K, l.N)
        if key not in cache:
            wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
            w0 = pkg.quantize(wb)
            del wb
            copies = max(2, -(-2 * l2 // l.weight_bytes))
            cache[key] = [w0] + [pkg.NVFP4Tensor(w0.codes.clone(), w0.scales.clone(),
                                                 w0.tensor_scale.clone())
                                 for _ in range(copies - 1)]
        ws_list = cache[key]
        x = torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        y = torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K), 16),
                         dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            for w in ws_list:
                pkg.gemm(x, w, y=y, stream=stream, workspace=ws)
        rounds = 10
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(rounds):
            for w in ws_list:
                pkg.gemm(x, w, y=y, stream=stream, workspace=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / (rounds * len(ws_list))
        b = l.weight_bytes + 2 * l.M * l.K + 2 * l.M * l.N
        n, k = pkg.imp_nvfp4_gemm_plan(l.M, l.N, l.K)
        skinny[f"M{l.M}_{l.K}x{l.N}"] = {"us": 1e3 * t, "GB/s": b / (t * 1e-3) / 1e9,
                                         "TFLOP/s": 2 * l.M * l.N * l.K / (t * 1e-3) / 1e12,
                                         "kernel": k, "launches": n}
    out["skinny_decode"] = skinny
    del cache
    # quantizer: the LM-head-sized weight
    l = synth.workload("decode_27b")[3]
    wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
    q = pkg.quantize(wb)
    times = []
    for i in range(args.warmup + 5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pkg.quantize(wb, out=q, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    t = statistics.median(times)
    qb = 2 * 2 * l.N * l.K + l.N * l.K // 2 + l.N * l.K // 16  # two reads of X + writes
    out["quantizer"] = {"shape": [l.N, l.K], "us": 1e3 * t, "GB/s": qb / (t * 1e-3) / 1e9,
                        "frac_of_hbm_peak": qb / (t * 1e-3) / 1e9 / hbm_peak}
    return out


def run_prefill_workload(args):
    """--workload prefill_27b: one step = the two prefill GEMMs (M = 2048) on
    the block-scaled FP4 tensor cores, X already quantized and W's scales in
    the atom layout; metric TFLOP/s.  e2e = imp_nvfp4_gemm from bf16 X copied
    from pinned host memory (quantization + W scale layout + GEMM) with Y
    copied back."""
    import torch

    import nvfp4_weight_quantized_02_gb300 as pkg

    if int(os.environ.get("RANK", "0")) != 0:
        return 0  # one GPU: the prefill workload is measured by rank 0 alone
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pkg.load()
    stream = torch.cuda.current_stream(dev)
    lins = synth.workload(args.workload)
    items = []
    for l in lins:
        wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        w = pkg.quantize(wb)
        del wb
        x = torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        items.append(dict(l=l, w=w, wm=pkg.prepare_mma(w), x=x, xq=pkg.quantize_mma(x),
                          y=torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev),
                          ws=torch.empty(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K),
                                         dtype=torch.uint8, device=dev),
                          ))
    flops = sum(2.0 * it["l"].M * it["l"].N * it["l"].K for it in items)

    def step():
        for it in items:
            pkg.gemm_fp4(it["xq"], it["wm"], y=it["y"], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    peak, kind = fp4_peak_tflops()
    value = flops / (ms * 1e-3) / 1e12
    pin_x = [torch.empty(it["x"].shape, dtype=torch.bfloat16, pin_memory=True).copy_(it["x"])
             for it in items]
    pin_y = [torch.empty(it["y"].shape, dtype=torch.bfloat16, pin_memory=True) for it in items]

    def e2e_step():
        for px, py, it in zip(pin_x, pin_y, items):
            it["x"].copy_(px, non_blocking=True)
            pkg.gemm(it["x"], it["w"], y=it["y"], stream=stream, workspace=it["ws"])
            py.copy_(it["y"], non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    line = {"metric": "prefill FP4 TFLOPS (block-scaled tcgen05 GEMM, M=2048)", "value": value,
            "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 x nvfp4, f32 accumulate, bf16 out", "data": "synthetic",
            "config": {"workload": args.workload,
                       "shapes_MxKxN": [[it["l"].M, it["l"].K, it["l"].N] for it in items]},
            "roofline": {"bound": "tensor", "kernel": "gemm_mxf4_kernel", "achieved": value,
                         "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                         "frac": value / peak, "traffic": None},
            "gpu_launches": args.steps * len(items), "clocks": clocks.summary(),
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": sum(p.numel() * 2 for p in pin_x),
                    "d2h_bytes_per_step": sum(p.numel() * 2 for p in pin_y)}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="decode workload (default decode_27b; <workload>:<name> for one problem)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload.startswith("prefill"):
        return run_prefill_workload(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
