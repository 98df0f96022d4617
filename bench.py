"""Benchmark of the NVFP4 linear layer on GB300.

One step is one decode pass of the 27B-class workload at M = 1, with the
dataflow of a decode layer: the up and gate projections (5120 -> 17408) read
the step's activation x, the down projection (17408 -> 5120) reads the gate
projection's output, the LM head (5120 -> 151936) reads the down
projection's output.  Each is Y = X W^T with an NVFP4 weight resident in
HBM, in the serving form (weights laid out once for the tensor cores by
imp_nvfp4_prepare_mma, then imp_nvfp4_gemm_mma per call).  The metric is the
rate at which the step streams its algorithmic bytes (NVFP4 weight bytes +
bf16 X and Y), in GB/s, next to the HBM roofline.  The weights of one step
(588 MB) exceed the 129 MB L2, so every step reads them from HBM.

Also reported (same JSON line): the same step on row-major weights through
imp_nvfp4_gemm and with unrelated inputs per projection, replayed as a CUDA
graph, the single 1024 x 1024 linear and the 0.6B-class layer (per call and
as a layer, weight copies rotated past L2), the per-M skinny decode rates,
the prefill GEMMs, the quantizer, and the spread (median, min, max) of every
rate over its repetitions.

The CPU baseline is the oracle (plain single-threaded C++: quantizer, fp64
matmul) timed on bounded samples of every workload.  ``--impl reference``
times only that oracle, as the reference arm.
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
L2_BYTES = 129 * 1024 * 1024


def call_bytes(l) -> int:
    """Algorithmic bytes of one call: NVFP4 weight + bf16 X and Y."""
    return l.weight_bytes + 2 * l.M * l.K + 2 * l.M * l.N


def step_bytes(lins) -> int:
    return sum(call_bytes(l) for l in lins)


def spread(vals):
    """median / min / max of a list of numbers."""
    return {"median": statistics.median(vals), "min": min(vals), "max": max(vals), "n": len(vals)}


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

def _cpu_jobs(max_rows: int):
    """(label, Linear, row sample) of every configuration of the workloads:
    configs 1 and 2 whole, config 3 and 4 on their first `max_rows` weight
    rows, config 5 on the 64-row sample of X (rows 32 i) against its first
    `max_rows` weight rows."""
    jobs = []
    for name in ("single_1k", "decode_0p6b", "decode_27b", "skinny_27b", "prefill_27b"):
        for l in synth.workload(name):
            jobs.append((f"{name}:{l.name}_M{l.M}", l, min(l.N, max_rows)))
    return jobs


def _prep_job(l, rows):
    import oracle
    wb = l.weight_bf16(0, rows)
    if l.M > 16:
        xs = l.act_bf16()[::32][:64]  # the 64-row sample
        return (l, wb, xs)
    return (l, wb, l.act_bf16())


def _run_job(job):
    """One pass of the oracle on a job: the quantizer on the sampled weight
    rows (tensor scale of the sample), then the matmul (for prefill, the
    activation quantized with the whole X's scale first).  Returns bytes of
    NVFP4 weight processed."""
    import oracle
    l, wb, x = job
    _, ts, _ = oracle.tensor_scale(wb)
    c, s = oracle.quantize_rows(wb, ts)
    oracle.reference_gemm(x, l.M, c, s, ts)
    return wb.shape[0] * (l.K // 2 + l.K // 16)


def cpu_oracle_sample(budget_s: float, max_rows: int = 128):
    """Time the oracle (quantizer + fp64 matmul, 1 thread) over every
    configuration's sample, repeated for about `budget_s` seconds.  Returns
    (GB/s of NVFP4 weight, seconds, description, per-config seconds)."""
    prepared = [(label, _prep_job(l, rows)) for label, l, rows in _cpu_jobs(max_rows)]
    per = {label: 0.0 for label, _ in prepared}
    done, passes, t0 = 0, 0, time.perf_counter()
    while True:
        for label, job in prepared:
            t1 = time.perf_counter()
            done += _run_job(job)
            per[label] += time.perf_counter() - t1
        passes += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    desc = (f"oracle quantizer + fp64 matmul (1 thread) on every configuration: configs 1-2 "
            f"whole, configs 3-4 on the first {max_rows} weight rows, config 5 on X rows 32 i "
            f"(i < 64) x the first {max_rows} weight rows; {passes} passes")
    return done / dt / 1e9, dt, desc, {k: v / passes for k, v in per.items()}


def _all_core_worker(args):
    part, max_rows, budget_s = args
    prepared = []
    for label, l, rows in _cpu_jobs(max_rows):
        r0 = min(part * rows, max(0, l.N - rows))
        wb = l.weight_bf16(r0, rows)
        x = l.act_bf16()[::32][:64] if l.M > 16 else l.act_bf16()
        prepared.append((l, wb, x))
    done, t0 = 0, time.perf_counter()
    while True:
        for job in prepared:
            done += _run_job(job)
        if time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0


def cpu_oracle_all_cores(budget_s: float, max_rows: int = 64):
    """The same oracle work as independent copies, one spawned process per
    core of this process's affinity mask, each on its own weight-row block
    (nothing is forked after the GPU was touched).  Returns (GB/s, cores,
    description)."""
    import multiprocessing as mp

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_all_core_worker, [(i, max_rows, budget_s) for i in range(cores)])
    gbs = sum(b / t for b, t in res) / 1e9
    desc = (f"oracle quantizer + fp64 matmul on every configuration, {cores} processes, each on "
            f"its own {max_rows}-row block of every weight, ~{budget_s:.0f} s")
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
    """The reference arm: the CPU oracle alone, on this host's cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    budget = max(0.5, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_sample(0.0, max_rows=16)
    gbs_all, per_step = [], []
    desc = ""
    for _ in range(args.steps):
        gbs, dt, desc, _ = cpu_oracle_sample(budget)
        per_step.append(dt)
        gbs_all.append(gbs)
    gbs = statistics.median(gbs_all)
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(per_step), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "M": 1,
                       "shapes_KxN": [[l.K, l.N] for l in synth.workload(args.workload)],
                       "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc, "spread": spread(gbs_all)},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def chain_inputs(lins, xs, ys):
    """The X each problem of a decode pass reads, in a decode layer's
    dataflow: gate reads up's x, down reads gate's output, the LM head reads
    down's output (when those problems are in the list and the widths
    match); every other problem reads its own synthetic X."""
    by = {l.name: i for i, l in enumerate(lins)}
    out = list(xs)
    for dst, src, kind in (("gate", "up", "x"), ("down", "gate", "y"), ("lm_head", "down", "y")):
        if dst in by and src in by:
            i, j = by[dst], by[src]
            width = lins[j].K if kind == "x" else lins[j].N
            if width == lins[i].K and lins[i].M == lins[j].M:
                out[i] = out[j] if kind == "x" else ys[j]
    return out


def layer_inputs_0p6b(lins, xs, ys):
    """The 0.6B-class layer's dataflow: q, k, v, gate and up read x; o reads
    q's output; down reads gate's output."""
    by = {l.name: i for i, l in enumerate(lins)}
    out = list(xs)
    for name in ("k", "v", "gate", "up"):
        out[by[name]] = xs[by["q"]]
    out[by["o"]] = ys[by["q"]]
    out[by["down"]] = ys[by["gate"]]
    return out


def event_pair():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def time_blocks(fn, n_per_block, blocks, stream):
    """Per-call µs of `blocks` blocks of `n_per_block` back-to-back calls."""
    import torch
    out = []
    for _ in range(blocks):
        e0, e1 = event_pair()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n_per_block):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(1e3 * e0.elapsed_time(e1) / n_per_block)
    return out


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
    hbm_peak, _, peak_kind = load_peaks()

    # ---- inputs resident in HBM (weights quantized and laid out on device; not timed)
    lins = synth.workload(args.workload)
    rows_w, weights, xs, ys = [], [], [], []
    for l in lins:
        wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        if args.weights == "fp8":
            w = pkg.fp8_quantize(wb)
        elif args.weights == "mxfp4":
            w = pkg.mxfp4_to_nvfp4(pkg.mxfp4_quantize(wb))
        else:
            w = pkg.quantize(wb)
        del wb
        rows_w.append(w)
        weights.append(w if args.weights == "fp8" else pkg.prepare_mma(w))
        xs.append(torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev))
        ys.append(torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev))
    chained = chain_inputs(lins, xs, ys)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # one workspace per problem, allocated once (the FP4 decode path's split
    # X, partial sums and counters)
    wss = [torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K),
                           pkg.imp_fp8_gemm_workspace_size(l.M, l.N, l.K), 16),
                       dtype=torch.uint8, device=dev) for l in lins]
    fp8 = args.weights == "fp8"
    plans = [pkg.imp_fp8_gemm_plan(l.M, l.N, l.K) if fp8 else pkg.imp_nvfp4_gemm_plan(l.M, l.N, l.K)
             for l in lins]
    call = pkg.gemm_fp8 if fp8 else pkg.gemm_mma
    use_chain = args.chain and not fp8

    def chain_of(ins, outs):
        """The step's calls as one decode chain (a call reading the previous
        call's output takes it from there)."""
        spec = []
        for i, (x, w, y) in enumerate(zip(ins, weights, outs)):
            g = [pkg.ImpNvfp4Group(w.c_struct(), y.data_ptr(), y.stride(0))]
            dep = i > 0 and x is outs[i - 1]
            spec.append((g, None if dep else x.data_ptr(), 0 if dep else x.stride(0)))
        return pkg.ChainLinks(spec)

    def run_chain(cl, ws, st):
        r = pkg.imp_nvfp4_gemm_chain(1, cl, status.data_ptr(), ws.data_ptr(), ws.numel(), st)
        if r != pkg.IMP_OK:
            raise pkg.ImpError(r, "imp_nvfp4_gemm_chain")

    if use_chain:
        step_chain = chain_of(chained, ys)
        chain_ws = torch.empty(pkg.imp_nvfp4_gemm_chain_workspace_size(1, step_chain),
                               dtype=torch.uint8, device=dev)
        if pkg.imp_nvfp4_gemm_chain_plan(1, step_chain) != 1:
            raise RuntimeError("the decode chain has no persistent plan for this workload")
    torch.cuda.synchronize()

    def step():
        if use_chain:
            run_chain(step_chain, chain_ws, pkg._stream_handle(stream))
            return
        for x, w, y, ws in zip(chained, weights, ys, wss):
            call(x, w, y=y, dev_status=status, stream=stream, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    bytes_step = step_bytes(lins)
    if fp8:  # one byte per weight, one tensor scale
        bytes_step = sum(l.N * l.K + 4 + 2 * l.M * (l.K + l.N) for l in lins)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        e0, e1 = event_pair()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        elapsed_ms = e0.elapsed_time(e1)
        # spread: ten more blocks of max(steps, 50) steps
        blocks = time_blocks(step, max(args.steps, 50), 10, stream)
        # the dominant call timed on its own (events around each call) >= 50 times,
        # on the stream it is launched on
        top = int(np.argmax([l.weight_bytes for l in lins]))
        per_call = {}
        for i, l in enumerate(lins):
            ts = []
            for _ in range(max(50, args.steps // 4)):
                a, b = event_pair()
                a.record(stream)
                call(chained[i], weights[i], y=ys[i], dev_status=status, stream=stream,
                     workspace=wss[i])
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            per_call[l.name] = [1e3 * a.elapsed_time(b) for a, b in ts]
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    if world > 1:
        dist.barrier()
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")
    ms_per_step = elapsed_ms / args.steps
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9

    # ---- e2e through the public API: every step copies its x in from pinned
    # host memory and its logits (the step's result) back.  As a serving loop
    # does, the copies run on a second stream (the copy engines) and overlap
    # the neighbouring steps' compute: two x buffers and two logits buffers,
    # each reused only after the step that holds it has finished with it.
    x0 = chained[0]
    pin_x = torch.empty(x0.shape, dtype=torch.bfloat16, pin_memory=True).copy_(x0)
    y_last = ys[-1]
    xin = [x0, torch.empty_like(x0)]
    logits = [y_last, torch.empty_like(y_last)]
    pin_y = [torch.empty(y_last.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    feeds = []
    for k in range(2):
        ins = [xin[k] if c is x0 else c for c in chained]
        outs = ys[:-1] + [logits[k]]
        feeds.append((ins, outs))
    copy_stream = torch.cuda.Stream(dev)

    feed_chains = [chain_of(ins, outs) for ins, outs in feeds] if use_chain else None

    def step_on(k):
        if use_chain:
            run_chain(feed_chains[k], chain_ws, pkg._stream_handle(stream))
            return
        ins, outs = feeds[k]
        for x, w, y, ws in zip(ins, weights, outs, wss):
            call(x, w, y=y, dev_status=status, stream=stream, workspace=ws)

    def e2e_run(n):
        """n steps; returns the elapsed ms between events on `stream`."""
        ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("h2d", "comp", "d2h")}
        a, b = event_pair()
        a.record(stream)
        copy_stream.wait_event(a)
        with torch.cuda.stream(copy_stream):
            for k in range(min(2, n)):
                xin[k].copy_(pin_x, non_blocking=True)
                ev["h2d"][k].record(copy_stream)
        for i in range(n):
            k = i % 2
            stream.wait_event(ev["h2d"][k])
            if i >= 2:
                stream.wait_event(ev["d2h"][k])  # logits[k] read back
            step_on(k)
            ev["comp"][k].record(stream)
            copy_stream.wait_event(ev["comp"][k])
            with torch.cuda.stream(copy_stream):
                pin_y[k].copy_(logits[k], non_blocking=True)
                ev["d2h"][k].record(copy_stream)
                if i + 2 < n:  # x of step i + 2 into the buffer step i is done with
                    xin[k].copy_(pin_x, non_blocking=True)
                    ev["h2d"][k].record(copy_stream)
        stream.wait_stream(copy_stream)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    e2e_run(max(args.warmup, 2))
    e2e_ms = max_over_ranks(e2e_run(args.steps) / args.steps, world, dev)
    e2e_value = world * bytes_step / (e2e_ms * 1e-3) / 1e9

    # ---- roofline of the dominant kernel: its call's bytes over the median
    # duration of the call timed alone (the call is the X split kernel + the
    # GEMV), and the same call launched back to back
    lt = lins[top]
    cbytes = (lambda l: l.N * l.K + 4 + 2 * l.M * (l.K + l.N)) if fp8 else call_bytes
    top_us = statistics.median(per_call[lt.name])
    achieved = cbytes(lt) / (top_us * 1e-6) / 1e9
    top_kernel = plans[top][1]
    traffic = None if args.weights != "nvfp4" else load_traffic(top_kernel, lt)
    b2b = time_blocks(lambda: call(chained[top], weights[top], y=ys[top],
                                   dev_status=status, stream=stream,
                                   workspace=wss[top]), 20, 5, stream)
    b2b_us = statistics.median(b2b)

    extra = {}
    if rank == 0 and not args.no_extra and args.weights == "nvfp4":
        extra = bench_extras(args, pkg, dev, stream, hbm_peak, lins, rows_w, weights, xs,
                             chained, ys, wss, status, step)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the extra measurements")

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"nvfp4": "nvfp4 weights, bf16 x/y, f32 accumulate",
                  "mxfp4": "mxfp4 weights (served in nvfp4 form), bf16 x/y, f32 accumulate",
                  "fp8": "fp8 e4m3 weights, bf16 x/y, f32 accumulate"}[args.weights],
        "data": "synthetic",
        "config": {"workload": args.workload, "M": 1, "shapes_KxN": [[l.K, l.N] for l in lins],
                   "bytes_per_step": bytes_step,
                   "dataflow": "decode layer: up and gate read x, down reads gate's output, "
                               "the LM head reads down's output",
                   "weights": {"nvfp4": "serving form (imp_nvfp4_prepare_mma once, "
                                        "imp_nvfp4_gemm_mma per call)",
                               "mxfp4": "MXFP4, converted once to NVFP4 form and prepared",
                               "fp8": "FP8 E4M3 row-major (imp_fp8_gemm per call)"}[args.weights],
                   "step_api": ("imp_nvfp4_gemm_chain, one launch per step" if use_chain else
                                "one imp_nvfp4_gemm_mma (fp8: imp_fp8_gemm) per call"),
                   "l2": "inputs larger than L2 (588 MB of weights per step)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm_peak": value / world / hbm_peak,
        "spread_us_per_step": spread(blocks),
        "per_call_us": {l.name: spread(per_call[l.name]) for l in lins},
        "per_call_gbs": {l.name: cbytes(l) / (statistics.median(per_call[l.name]) * 1e-6) / 1e9
                         for l in lins},
        "roofline": {"bound": "hbm", "kernel": f"{top_kernel} ({lt.name} {lt.K}x{lt.N})",
                     "achieved": achieved, "peak": hbm_peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "bytes_per_launch": cbytes(lt),
                     "back_to_back": {"us_per_launch": b2b_us,
                                      "achieved": cbytes(lt) / (b2b_us * 1e-6) / 1e9,
                                      "frac": cbytes(lt) / (b2b_us * 1e-6) / 1e9 / hbm_peak}},
        "gpu_launches": args.steps * (1 if use_chain else sum(n for n, _ in plans)),
        "kernels": ({"step": {"kernel": "gemv_f4c_kernel", "launches_per_step": 1}} if use_chain else
                    {l.name: {"kernel": k, "launches_per_call": n} for l, (n, k) in zip(lins, plans)}),
        "clocks": clocks.summary(),
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": pin_x.numel() * 2,
                "d2h_bytes_per_step": pin_y[0].numel() * 2,
                "copies": "second stream, overlapping the neighbouring steps (two x and two "
                          "logits buffers)"},
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu_baseline and args.weights == "nvfp4":
        gbs, dt, desc, per = cpu_oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": dt,
                                "per_config_ms": {k: 1e3 * v for k, v in per.items()}}
        if world == 1:
            try:
                gbs, cores, desc = cpu_oracle_all_cores(args.cpu_seconds)
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


def rotated_copies(pkg, w, copies):
    """`copies` device copies of a weight (the first is `w`)."""
    return [w] + [pkg.NVFP4Tensor(w.codes.clone(), w.scales.clone(), w.tensor_scale.clone(),
                                  layout=w.layout, shape=(w.rows, w.K)) for _ in range(copies - 1)]


def bench_small_configs(pkg, dev, stream, hbm_peak, status):
    """Configs 1 and 2 (launch-bound shapes): per call and, for the 0.6B-class
    layer, as the seven calls of one layer in its dataflow -- eagerly and
    replayed as a CUDA graph.  Weights rotate over enough copies to exceed
    three times the L2, so every call reads its weight from HBM."""
    import torch

    out = {}
    for name in ("single_1k", "decode_0p6b"):
        lins = synth.workload(name)
        base = []
        for l in lins:
            wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
            base.append(pkg.prepare_mma(pkg.quantize(wb)))
            del wb
        layer_bytes = step_bytes(lins)
        ncopy = -(-3 * L2_BYTES // layer_bytes) + 1
        copies = [rotated_copies(pkg, w, ncopy) for w in base]  # [problem][copy]
        xs = [torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
              for l in lins]
        ys = [torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev) for l in lins]
        wss = [torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K), 16),
                           dtype=torch.uint8, device=dev) for l in lins]
        ins = layer_inputs_0p6b(lins, xs, ys) if name == "decode_0p6b" else xs
        res = {"weight_copies": ncopy, "calls": {}}
        for i, l in enumerate(lins):
            k = [0]

            def one(i=i, k=k):
                pkg.gemm_mma(ins[i], copies[i][k[0] % ncopy], y=ys[i], dev_status=status,
                             stream=stream, workspace=wss[i])
                k[0] += 1
            for _ in range(ncopy):
                one()
            ts = time_blocks(one, ncopy, 10, stream)
            med = statistics.median(ts)
            res["calls"][f"{l.name}_{l.K}x{l.N}"] = {
                "us": spread(ts), "GB/s": call_bytes(l) / (med * 1e-6) / 1e9,
                "frac_of_hbm_peak": call_bytes(l) / (med * 1e-6) / 1e9 / hbm_peak,
                "kernel": pkg.imp_nvfp4_gemm_plan(l.M, l.N, l.K)[1]}
        if len(lins) > 1:
            k = [0]

            def layer(k=k):
                c = k[0] % ncopy
                for i in range(len(lins)):
                    pkg.gemm_mma(ins[i], copies[i][c], y=ys[i], dev_status=status,
                                 stream=stream, workspace=wss[i])
                k[0] += 1
            for _ in range(ncopy):
                layer()
            ts = time_blocks(layer, ncopy, 10, stream)
            med = statistics.median(ts)
            res["layer_eager"] = {"us": spread(ts), "GB/s": layer_bytes / (med * 1e-6) / 1e9,
                                  "sum_of_calls_us": sum(v["us"]["median"]
                                                         for v in res["calls"].values())}
            # the layer captured once per weight copy and replayed
            try:
                cap = torch.cuda.Stream(dev)
                cap.wait_stream(stream)
                graphs = []
                for c in range(ncopy):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=cap):
                        for i in range(len(lins)):
                            pkg.gemm_mma(ins[i], copies[i][c], y=ys[i], dev_status=status,
                                         stream=cap, workspace=wss[i])
                    graphs.append(g)
                torch.cuda.synchronize()
                gs = torch.cuda.current_stream(dev)
                for g in graphs:
                    g.replay()
                ts = []
                for _ in range(10):
                    a, b = event_pair()
                    torch.cuda.synchronize()
                    a.record(gs)
                    for g in graphs:
                        g.replay()
                    b.record(gs)
                    torch.cuda.synchronize()
                    ts.append(1e3 * a.elapsed_time(b) / ncopy)
                med = statistics.median(ts)
                res["layer_graph"] = {"us": spread(ts), "GB/s": layer_bytes / (med * 1e-6) / 1e9}
                del graphs
            except Exception as e:  # report, do not fail the line
                res["layer_graph"] = {"error": str(e)[:200]}
        if name == "decode_0p6b":
            res.update(bench_grouped_layer(pkg, dev, stream, status, lins, copies, ncopy, ins,
                                           ys, layer_bytes))
        out[name] = res
        del copies, base
    return out


def bench_grouped_layer(pkg, dev, stream, status, lins, copies, ncopy, ins, ys, layer_bytes):
    """The 0.6B-class layer as four calls: q/k/v grouped, o, gate/up grouped,
    down (8 kernels instead of 14), eagerly and replayed as CUDA graphs."""
    import torch

    by = {l.name: i for i, l in enumerate(lins)}
    x = ins[by["q"]]
    groups = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
    wsz = 16
    for g in groups:
        wsz = max(wsz, pkg.imp_nvfp4_gemm_grouped_workspace_size(1, lins[by[g[0]]].K,
                                                                 [lins[by[n]].N for n in g]))
    ws = torch.empty(wsz, dtype=torch.uint8, device=dev)
    launches = sum(pkg.imp_nvfp4_gemm_grouped_plan(1, lins[by[g[0]]].K,
                                                   [lins[by[n]].N for n in g])[0] for g in groups)

    def calls(c, st):
        for g in groups:
            i0 = by[g[0]]
            pkg.gemm_grouped(x if len(g) > 1 else ins[i0], [copies[by[n]][c] for n in g],
                             ys=[ys[by[n]] for n in g], dev_status=status, stream=st,
                             workspace=ws)
    k = [0]

    def layer():
        calls(k[0] % ncopy, stream)
        k[0] += 1
    for _ in range(ncopy):
        layer()
    res = {}
    ts = time_blocks(layer, ncopy, 10, stream)
    med = statistics.median(ts)
    res["layer_grouped_eager"] = {"us": spread(ts), "GB/s": layer_bytes / (med * 1e-6) / 1e9,
                                  "launches": launches}
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graphs = []
        for c in range(ncopy):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                calls(c, cap)
            graphs.append(g)
        torch.cuda.synchronize()
        gs = torch.cuda.current_stream(dev)
        for g in graphs:
            g.replay()
        ts = []
        for _ in range(10):
            a, b = event_pair()
            torch.cuda.synchronize()
            a.record(gs)
            for g in graphs:
                g.replay()
            b.record(gs)
            torch.cuda.synchronize()
            ts.append(1e3 * a.elapsed_time(b) / ncopy)
        med = statistics.median(ts)
        res["layer_grouped_graph"] = {"us": spread(ts), "GB/s": layer_bytes / (med * 1e-6) / 1e9,
                                      "launches": launches}
        del graphs
    except Exception as e:  # report, do not fail the line
        res["layer_grouped_graph"] = {"error": str(e)[:200]}
    # the same four calls as one decode chain (imp_nvfp4_gemm_chain: one
    # launch; o and down read their predecessors' outputs)
    try:
        def links_for(c):
            spec = []
            for g in groups:
                i0 = by[g[0]]
                gl = [pkg.ImpNvfp4Group(copies[by[n]][c].c_struct(), ys[by[n]].data_ptr(),
                                        ys[by[n]].stride(0)) for n in g]
                dep = len(g) == 1 and ins[i0] is ys[by[groups[groups.index(g) - 1][0]]]
                xx = x if len(g) > 1 else ins[i0]
                spec.append((gl, None if dep else xx.data_ptr(), 0 if dep else xx.stride(0)))
            return pkg.ChainLinks(spec)
        cls = [links_for(c) for c in range(ncopy)]
        cws = torch.empty(max(pkg.imp_nvfp4_gemm_chain_workspace_size(1, cl) for cl in cls),
                          dtype=torch.uint8, device=dev)
        sh = pkg._stream_handle(stream)
        kc = [0]

        def chain_layer():
            st = pkg.imp_nvfp4_gemm_chain(1, cls[kc[0] % ncopy], status.data_ptr(),
                                          cws.data_ptr(), cws.numel(), sh)
            if st != pkg.IMP_OK:
                raise pkg.ImpError(st, "imp_nvfp4_gemm_chain")
            kc[0] += 1
        for _ in range(ncopy):
            chain_layer()
        ts = time_blocks(chain_layer, ncopy, 10, stream)
        med = statistics.median(ts)
        res["layer_chain"] = {"us": spread(ts), "GB/s": layer_bytes / (med * 1e-6) / 1e9,
                              "launches": 1,
                              "persistent_launch": pkg.imp_nvfp4_gemm_chain_plan(1, cls[0]) == 1}
    except Exception as e:  # report, do not fail the line
        res["layer_chain"] = {"error": str(e)[:200]}
    return res


def bench_weight_formats(args, pkg, dev, stream, hbm_peak, lins, status):
    """The decode step (same shapes and dataflow) on the README's other
    weight formats: MXFP4 weights converted once to the NVFP4 form (so the
    step streams the same 0.5625 B per weight as the NVFP4 step; the MXFP4
    format itself is 0.53125 B), and FP8 E4M3 weights (1 B per weight)
    through imp_fp8_gemm."""
    import torch

    out = {}
    n = max(args.steps, 50)
    mx_w, f8_w = [], []
    for l in lins:
        wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        mx_w.append(pkg.prepare_mma(pkg.mxfp4_to_nvfp4(pkg.mxfp4_quantize(wb, dev_status=status),
                                                       dev_status=status)))
        f8_w.append(pkg.fp8_quantize(wb, dev_status=status))
        del wb
    xs = [torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev) for l in lins]
    ys = [torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev) for l in lins]
    chained = chain_inputs(lins, xs, ys)
    wss = [torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K),
                           pkg.imp_fp8_gemm_workspace_size(l.M, l.N, l.K), 16),
                       dtype=torch.uint8, device=dev) for l in lins]
    torch.cuda.synchronize()

    def mx_step():
        for x, w, y, ws in zip(chained, mx_w, ys, wss):
            pkg.gemm_mma(x, w, y=y, dev_status=status, stream=stream, workspace=ws)

    def f8_step():
        for x, w, y, ws in zip(chained, f8_w, ys, wss):
            pkg.gemm_fp8(x, w, y=y, dev_status=status, stream=stream, workspace=ws)

    mx_bytes = sum(l.N * l.K // 2 + l.N * l.K // 32 + 2 * l.M * (l.K + l.N) for l in lins)
    nv_bytes = step_bytes(lins)
    f8_bytes = sum(l.N * l.K + 4 + 2 * l.M * (l.K + l.N) for l in lins)
    for name, fn, nbytes, extra in (
            ("decode_mxfp4_weights", mx_step, nv_bytes,
             {"weights": "MXFP4 (OCP MX) quantized, converted once to NVFP4 form and prepared",
              "mxfp4_format_bytes_per_step": mx_bytes}),
            ("decode_fp8_weights", f8_step, f8_bytes,
             {"weights": "FP8 E4M3, one fp32 tensor scale, row-major (imp_fp8_gemm)",
              "kernels": [pkg.imp_fp8_gemm_plan(l.M, l.N, l.K) for l in lins]})):
        for _ in range(args.warmup):
            fn()
        ts = time_blocks(fn, n, 10, stream)
        med = statistics.median(ts)
        out[name] = {"us_per_step": spread(ts), "bytes_per_step": nbytes,
                     "GB/s": nbytes / (med * 1e-6) / 1e9,
                     "frac_of_hbm_peak": nbytes / (med * 1e-6) / 1e9 / hbm_peak, **extra}
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the weight-format steps")
    del mx_w, f8_w
    return out


def bench_prefill(args, pkg, dev, stream):
    """Prefill GEMMs (M = 2048): the block-scaled FP4 tensor-core GEMM alone
    (X already quantized, W in the MMA layout) and the whole imp_nvfp4_gemm
    call (X quantization + GEMM)."""
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
                         ("imp_nvfp4_gemm_mma", lambda: pkg.gemm_mma(x, wm, y=y, stream=stream,
                                                                     workspace=ws))):
            for _ in range(args.warmup):
                fn()
            ts = time_blocks(fn, 10, 6, stream)
            t = statistics.median(ts)
            tf = flops / (t * 1e-6) / 1e12
            out[name] = {"us": spread(ts), "TFLOP/s": tf, "frac_of_fp4_peak": tf / peak}
        res[f"M{l.M}_{l.K}x{l.N}"] = out
        del w, wm, x, xq, y, ws, wsf
    res["fp4_peak_tflops"] = peak
    res["fp4_peak_kind"] = f"{kind} bf16 x 6 (nominal fp4:bf16 ratio)"
    res["mlp_27b"] = bench_prefill_mlp(args, pkg, dev, stream, peak)
    return res


def bench_prefill_mlp(args, pkg, dev, stream, peak):
    """The 27B-class MLP at M = 2048 (X 2048 x 5120 -> gate/up 17408 ->
    SwiGLU -> down 5120): fused = imp_nvfp4_gemm_swiglu (X quantization +
    gate/up GEMM with the activation and the amax of h in its epilogue) +
    imp_nvfp4_quantize_mma_amax (one read of h) + the down GEMM; unfused =
    imp_nvfp4_gemm_mma for gate and for up + the two-pass quantizer of h +
    the down GEMM (the activation itself, which the library has no separate
    kernel for, left out: the unfused figure is a lower bound)."""
    import torch

    lg = [l for l in synth.workload("prefill_27b") if l.K == 5120][0]
    ld = [l for l in synth.workload("prefill_27b") if l.K == 17408][0]
    lu = synth.Linear("up_27b", lg.M, lg.K, lg.N, 41, w_dist=synth.DIST_STUDENT_T4, w_scale=0.02,
                      zero_block_p=0.001)
    mk = lambda l: pkg.prepare_mma(pkg.quantize(  # noqa: E731
        torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)))
    wg, wu, wd = mk(lg), mk(lu), mk(ld)
    x = torch.from_numpy(lg.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
    h = torch.empty((lg.M, lg.N), dtype=torch.bfloat16, device=dev)
    hu = torch.empty_like(h)
    amax = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.empty((ld.M, ld.N), dtype=torch.bfloat16, device=dev)
    wss = torch.empty(pkg.imp_nvfp4_gemm_swiglu_workspace_size(lg.M, lg.N, lg.K), dtype=torch.uint8,
                      device=dev)
    wsg = torch.empty(pkg.imp_nvfp4_gemm_workspace_size(lg.M, lg.N, lg.K), dtype=torch.uint8,
                      device=dev)
    hq = pkg.quantize_mma(h)

    def fused():
        pkg.gemm_swiglu(x, wg, wu, h=h, h_amax=amax, stream=stream, workspace=wss)
        q = pkg.quantize_mma_amax(h, amax, stream=stream)
        pkg.gemm_fp4(q, wd, y=y, stream=stream)

    def unfused():
        pkg.gemm_mma(x, wg, y=h, stream=stream, workspace=wsg)
        pkg.gemm_mma(x, wu, y=hu, stream=stream, workspace=wsg)
        q = pkg.quantize_mma(h, stream=stream)
        pkg.gemm_fp4(q, wd, y=y, stream=stream)

    flops = 2.0 * lg.M * lg.K * lg.N * 2 + 2.0 * ld.M * ld.K * ld.N
    out = {"shapes": {"x": [lg.M, lg.K], "gate_up_N": lg.N, "down_N": ld.N}, "flop": flops}
    for name, fn in (("fused", fused), ("unfused_without_activation", unfused)):
        for _ in range(args.warmup):
            fn()
        ts = time_blocks(fn, 5, 6, stream)
        t = statistics.median(ts)
        out[name] = {"us": spread(ts), "TFLOP/s": flops / (t * 1e-6) / 1e12,
                     "frac_of_fp4_peak": flops / (t * 1e-6) / 1e12 / peak}
    del wg, wu, wd, x, h, hu, y, wss, wsg, hq
    return out


def bench_extras(args, pkg, dev, stream, hbm_peak, lins, rows_w, weights, xs, chained, ys, wss,
                 status, step):
    """Variants of the step, configs 1 and 2, skinny M, prefill, quantizer."""
    import torch

    bytes_step = step_bytes(lins)

    def rate(ts):
        med = statistics.median(ts)
        return {"us_per_step": spread(ts), "GB/s": bytes_step / (med * 1e-6) / 1e9,
                "frac_of_hbm_peak": bytes_step / (med * 1e-6) / 1e9 / hbm_peak}

    out = {}
    n = max(args.steps, 50)

    # the step on row-major weights (no layout transform) through imp_nvfp4_gemm
    def rows_step():
        for x, w, y, ws in zip(chained, rows_w, ys, wss):
            pkg.gemm(x, w, y=y, dev_status=status, stream=stream, workspace=ws)
    for _ in range(args.warmup):
        rows_step()
    out["decode_row_major_weights"] = rate(time_blocks(rows_step, n, 10, stream))

    # the step with an unrelated synthetic X per projection (no dataflow: every
    # X is read from HBM, not from the previous call's output in L2)
    def indep_step():
        for x, w, y, ws in zip(xs, weights, ys, wss):
            pkg.gemm_mma(x, w, y=y, dev_status=status, stream=stream, workspace=ws)
    for _ in range(args.warmup):
        indep_step()
    out["decode_independent_inputs"] = rate(time_blocks(indep_step, n, 10, stream))

    # the step with up and gate as one grouped call (one split of x, one
    # weight stream over both weights' tiles)
    by = {l.name: i for i, l in enumerate(lins)}
    if "up" in by and "gate" in by:
        iu, ig = by["up"], by["gate"]
        gws = torch.empty(pkg.imp_nvfp4_gemm_grouped_workspace_size(
            1, lins[iu].K, [lins[iu].N, lins[ig].N]), dtype=torch.uint8, device=dev)

        def grouped_step():
            pkg.gemm_grouped(chained[iu], [weights[iu], weights[ig]], ys=[ys[iu], ys[ig]],
                             dev_status=status, stream=stream, workspace=gws)
            for i, (x, w, y, ws) in enumerate(zip(chained, weights, ys, wss)):
                if i not in (iu, ig):
                    pkg.gemm_mma(x, w, y=y, dev_status=status, stream=stream, workspace=ws)
        for _ in range(args.warmup):
            grouped_step()
        out["decode_grouped_up_gate"] = rate(time_blocks(grouped_step, n, 10, stream))

        # the layer's true MLP dataflow: gate and up grouped, the down
        # projection on silu(gate) * up (formed in its X split), the LM head
        # on down's output
        if "down" in by and lins[by["down"]].K == lins[ig].N:
            idn = by["down"]
            rest = [i for i in range(len(lins)) if i not in (iu, ig, idn)]

            def swiglu_step():
                pkg.gemm_grouped(chained[iu], [weights[ig], weights[iu]], ys=[ys[ig], ys[iu]],
                                 dev_status=status, stream=stream, workspace=gws)
                pkg.gemm_mma_swiglu(ys[ig], ys[iu], weights[idn], y=ys[idn], dev_status=status,
                                    stream=stream, workspace=wss[idn])
                for i in rest:
                    pkg.gemm_mma(chained[i], weights[i], y=ys[i], dev_status=status,
                                 stream=stream, workspace=wss[i])
            for _ in range(args.warmup):
                swiglu_step()
            out["decode_swiglu_mlp"] = dict(
                rate(time_blocks(swiglu_step, n, 10, stream)),
                dataflow="gate and up grouped on x; down on silu(gate) * up; LM head on down")
            # the same as one decode-chain launch (x_swiglu link)
            if "lm_head" in by and rest == [by["lm_head"]]:
                il = by["lm_head"]
                g2 = [pkg.ImpNvfp4Group(weights[j].c_struct(), ys[j].data_ptr(), ys[j].stride(0))
                      for j in (ig, iu)]
                cl = pkg.ChainLinks([
                    (g2, chained[iu].data_ptr(), chained[iu].stride(0)),
                    ([pkg.ImpNvfp4Group(weights[idn].c_struct(), ys[idn].data_ptr(),
                                        ys[idn].stride(0))], None, 0, 1),
                    ([pkg.ImpNvfp4Group(weights[il].c_struct(), ys[il].data_ptr(),
                                        ys[il].stride(0))], None, 0)])
                cws = torch.empty(pkg.imp_nvfp4_gemm_chain_workspace_size(1, cl),
                                  dtype=torch.uint8, device=dev)
                sh = pkg._stream_handle(stream)

                def swiglu_chain():
                    st = pkg.imp_nvfp4_gemm_chain(1, cl, status.data_ptr(), cws.data_ptr(),
                                                  cws.numel(), sh)
                    if st != pkg.IMP_OK:
                        raise pkg.ImpError(st, "imp_nvfp4_gemm_chain")
                for _ in range(args.warmup):
                    swiglu_chain()
                out["decode_swiglu_mlp_chain"] = dict(
                    rate(time_blocks(swiglu_chain, n, 10, stream)), launches_per_step=1,
                    persistent_launch=pkg.imp_nvfp4_gemm_chain_plan(1, cl) == 1)
                del cws
        del gws

    # the step as one decode chain (imp_nvfp4_gemm_chain: one persistent
    # launch; down and the LM head wait for their X, gate keeps up's split X)
    try:
        spec = []
        for i, (x, w, y) in enumerate(zip(chained, weights, ys)):
            g = [pkg.ImpNvfp4Group(w.c_struct(), y.data_ptr(), y.stride(0))]
            dep = i > 0 and x is ys[i - 1]
            spec.append((g, None if dep else x.data_ptr(), 0 if dep else x.stride(0)))
        cl = pkg.ChainLinks(spec)
        cws = torch.empty(pkg.imp_nvfp4_gemm_chain_workspace_size(1, cl), dtype=torch.uint8,
                          device=dev)
        sh = pkg._stream_handle(stream)

        def chain_step():
            st = pkg.imp_nvfp4_gemm_chain(1, cl, status.data_ptr(), cws.data_ptr(), cws.numel(),
                                          sh)
            if st != pkg.IMP_OK:
                raise pkg.ImpError(st, "imp_nvfp4_gemm_chain")
        for _ in range(args.warmup):
            chain_step()
        out["decode_chain"] = dict(rate(time_blocks(chain_step, n, 10, stream)),
                                   persistent_launch=pkg.imp_nvfp4_gemm_chain_plan(1, cl) == 1,
                                   launches_per_step=1)
        del cws
    except Exception as e:  # report, do not fail the benchmark line
        out["decode_chain"] = {"error": str(e)[:200]}

    # the step replayed as one CUDA graph (programmatic dependent launch kept)
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for x, w, y, ws in zip(chained, weights, ys, wss):
                pkg.gemm_mma(x, w, y=y, dev_status=status, stream=cap, workspace=ws)
        torch.cuda.synchronize()
        gs = torch.cuda.current_stream(dev)
        for _ in range(args.warmup):
            graph.replay()
        out["decode_graph_replay"] = rate(time_blocks(graph.replay, n, 10, gs))
        del graph
    except Exception as e:  # report, do not fail the benchmark line
        out["decode_graph_replay"] = {"error": str(e)[:200]}

    out.update(bench_weight_formats(args, pkg, dev, stream, hbm_peak, lins, status))
    out["small_configs"] = bench_small_configs(pkg, dev, stream, hbm_peak, status)
    out["prefill"] = bench_prefill(args, pkg, dev, stream)

    # Skinny M: back-to-back calls cycling through copies of W whose total
    # exceeds L2 twice over, so each call reads its weight from HBM.
    skinny = {}
    cache = {}
    for l in synth.workload("skinny_27b"):
        key = (l.K, l.N)
        if key not in cache:
            wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
            w0 = pkg.quantize(wb)
            del wb
            cache[key] = rotated_copies(pkg, pkg.prepare_mma(w0), max(2, -(-2 * L2_BYTES // l.weight_bytes)))
            del w0
        wl = cache[key]
        x = torch.from_numpy(l.act_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
        y = torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K), 16),
                         dtype=torch.uint8, device=dev)
        k = [0]

        def one(k=k, wl=wl, x=x, y=y, ws=ws):
            pkg.gemm_mma(x, wl[k[0] % len(wl)], y=y, dev_status=status, stream=stream,
                         workspace=ws)
            k[0] += 1
        for _ in range(len(wl) * 2):
            one()
        ts = time_blocks(one, len(wl) * 5, 10, stream)
        t = statistics.median(ts)
        nk, kern = pkg.imp_nvfp4_gemm_plan(l.M, l.N, l.K)
        skinny[f"M{l.M}_{l.K}x{l.N}"] = {"us": spread(ts), "GB/s": call_bytes(l) / (t * 1e-6) / 1e9,
                                         "frac_of_hbm_peak": call_bytes(l) / (t * 1e-6) / 1e9 / hbm_peak,
                                         "TFLOP/s": 2 * l.M * l.N * l.K / (t * 1e-6) / 1e12,
                                         "kernel": kern, "launches": nk}
    out["skinny_decode"] = skinny

    # The step's 50 MB projections (M = 1) one call after another, each call
    # on another copy of its weight (the copies exceed L2 twice over, so every
    # call streams its weight from HBM): a call's cost inside a stream of
    # calls, without event records between them.
    b2b, seen = {}, set()
    for i, l in enumerate(lins):
        if l.weight_bytes > L2_BYTES // 2 or (l.K, l.N) in seen:
            continue
        seen.add((l.K, l.N))
        wl = rotated_copies(pkg, weights[i], max(2, -(-2 * L2_BYTES // l.weight_bytes)))
        k = [0]

        def one(i=i, k=k, wl=wl):
            pkg.gemm_mma(chained[i], wl[k[0] % len(wl)], y=ys[i], dev_status=status,
                         stream=stream, workspace=wss[i])
            k[0] += 1
        for _ in range(len(wl) * 2):
            one()
        ts = time_blocks(one, len(wl) * 5, 10, stream)
        t = statistics.median(ts)
        b2b[f"{l.name}_{l.K}x{l.N}"] = {"us": spread(ts), "GB/s": call_bytes(l) / (t * 1e-6) / 1e9,
                                        "frac_of_hbm_peak": call_bytes(l) / (t * 1e-6) / 1e9 / hbm_peak,
                                        "weight_copies": len(wl)}
        del wl
    out["per_call_back_to_back"] = b2b
    del cache

    # quantizer: the LM-head-sized weight (two reads of X + codes and scales written)
    l = lins[-1]
    wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
    q = pkg.quantize(wb)
    for _ in range(args.warmup):
        pkg.quantize(wb, out=q, stream=stream)
    ts = time_blocks(lambda: pkg.quantize(wb, out=q, stream=stream), 1, 20, stream)
    t = statistics.median(ts)
    qb = 2 * 2 * l.N * l.K + l.N * l.K // 2 + l.N * l.K // 16
    out["quantizer"] = {"shape": [l.N, l.K], "us": spread(ts), "GB/s": qb / (t * 1e-6) / 1e9,
                        "frac_of_hbm_peak": qb / (t * 1e-6) / 1e9 / hbm_peak}
    del wb, q
    return out


def run_prefill_workload(args):
    """--workload prefill_27b: one step = the two prefill GEMMs (M = 2048) on
    the block-scaled FP4 tensor cores, X already quantized and W in the MMA
    layout; metric TFLOP/s.  e2e = imp_nvfp4_gemm_mma from bf16 X copied from
    pinned host memory (X quantization + GEMM) with Y copied back."""
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
        items.append(dict(l=l, wm=pkg.prepare_mma(w), x=x, xq=pkg.quantize_mma(x),
                          y=torch.empty((l.M, l.N), dtype=torch.bfloat16, device=dev),
                          ws=torch.empty(pkg.imp_nvfp4_gemm_workspace_size(l.M, l.N, l.K),
                                         dtype=torch.uint8, device=dev)))
        del w
    flops = sum(2.0 * it["l"].M * it["l"].N * it["l"].K for it in items)

    def step():
        for it in items:
            pkg.gemm_fp4(it["xq"], it["wm"], y=it["y"], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        e0, e1 = event_pair()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        blocks = time_blocks(step, max(args.steps, 10), 10, stream)
    ms = e0.elapsed_time(e1) / args.steps
    peak, kind = fp4_peak_tflops()
    value = flops / (ms * 1e-3) / 1e12
    pin_x = [torch.empty(it["x"].shape, dtype=torch.bfloat16, pin_memory=True).copy_(it["x"])
             for it in items]
    pin_y = [torch.empty(it["y"].shape, dtype=torch.bfloat16, pin_memory=True) for it in items]

    def e2e_step():
        for px, py, it in zip(pin_x, pin_y, items):
            it["x"].copy_(px, non_blocking=True)
            pkg.gemm_mma(it["x"], it["wm"], y=it["y"], stream=stream, workspace=it["ws"])
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
    n_launch = sum(pkg.imp_nvfp4_gemm_plan(it["l"].M, it["l"].N, it["l"].K)[0] for it in items)
    line = {"metric": "prefill FP4 TFLOPS (block-scaled tcgen05 GEMM, M=2048)", "value": value,
            "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 x nvfp4, f32 accumulate, bf16 out", "data": "synthetic",
            "config": {"workload": args.workload,
                       "shapes_MxKxN": [[it["l"].M, it["l"].K, it["l"].N] for it in items]},
            "spread_ms_per_step": spread([b / 1e3 for b in blocks]),
            "roofline": {"bound": "tensor", "kernel": "gemm_mxf4_kernel", "achieved": value,
                         "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                         "frac": value / peak, "traffic": None},
            "gpu_launches": args.steps * len(items), "clocks": clocks.summary(),
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": sum(p.numel() * 2 for p in pin_x),
                    "d2h_bytes_per_step": sum(p.numel() * 2 for p in pin_y),
                    "gpu_launches_per_step": n_launch}}
    print(json.dumps(line))
    return 0


def run_quantizer_workload(args):
    """--workload quantizer: one step = the NVFP4 quantizer (global amax pass,
    block encode pass) on the 27B-class LM-head weight (151936 x 5120 bf16);
    metric GB/s of its algorithmic bytes (X read twice, codes and scales
    written)."""
    import torch

    import nvfp4_weight_quantized_02_gb300 as pkg

    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pkg.load()
    stream = torch.cuda.current_stream(dev)
    l = [w for w in synth.workload("decode_27b") if w.name == "lm_head"][0]
    wb = torch.from_numpy(l.weight_bf16().view(np.int16)).view(torch.bfloat16).to(dev)
    q = pkg.NVFP4Tensor.empty(l.N, l.K, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    step = lambda: pkg.quantize(wb, out=q, dev_status=status, stream=stream)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        e0, e1 = event_pair()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        blocks = time_blocks(step, max(args.steps, 5), 10, stream)
    assert int(status.item()) == 0
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = 2 * 2 * l.N * l.K + l.N * l.K // 2 + l.N * l.K // 16
    hbm_peak, _, peak_kind = load_peaks()
    value = nbytes / (ms * 1e-3) / 1e9
    line = {"metric": "NVFP4 quantizer GB/s (two passes, bit-exact)", "value": value,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, nvfp4 out", "data": "synthetic",
            "config": {"workload": "quantizer", "shape": [l.N, l.K]},
            "spread_ms_per_step": spread([b / 1e3 for b in blocks]),
            "roofline": {"bound": "hbm", "kernel": "amax_partial_kernel + encode_kernel",
                         "achieved": value, "peak": hbm_peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": value / hbm_peak, "traffic": None},
            "gpu_launches": 2 * args.steps, "clocks": clocks.summary()}
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
    ap.add_argument("--chain", action="store_true",
                    help="run the decode step as one decode-chain launch (imp_nvfp4_gemm_chain)")
    ap.add_argument("--weights", choices=["nvfp4", "mxfp4", "fp8"], default="nvfp4",
                    help="weight format of the decode step (mxfp4: converted once to the NVFP4 "
                         "form; fp8: E4M3 with one tensor scale)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload.startswith("prefill"):
        return run_prefill_workload(args)
    if args.workload == "quantizer":
        return run_quantizer_workload(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
