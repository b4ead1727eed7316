#!/usr/bin/env python
"""Benchmark of the per-decode-step token sampler.

One step = one sampling call over the whole batch (load, penalties,
temperature, top-k/top-p, min-p, pick, optional probs/logprobs). Default
workload: N=64 rows, V=128000 bf16 logits ~ 2*N(0,1) with one +12 spike per
row; 32 rows T=0.8, 16 rows top_p=0.9 + top_k=50, 16 greedy; token ids only.

Prints one JSON line (rank 0). Our arm: steps replayed from a CUDA graph over
rotating input copies larger than L2, timed with CUDA events on the launch
stream; `e2e` through the host-buffer C entry point; `roofline` for the row
kernel; `cpu_baseline` = the CPU oracle on a bounded sample. `--impl
reference` times the CPU oracle itself (the only reference this sampler has).
Several GPUs run independent replicas (rows are independent: no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "sampled rows/s and HBM GB/s vs ~8 TB/s at N=64 V=128000 bf16, mixed params"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
KERNEL_DIR = os.path.join(ROOT, "decode_step_token_gb300", "csrc")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(KERNEL_DIR)):
        if not f.endswith((".cu", ".cuh")):
            continue
        with open(os.path.join(KERNEL_DIR, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def describe(batch) -> str:
    if batch.name == "mixed":
        return ("mixed: N=64 V=128000 bf16 logits 2*N(0,1) + 12 at one token per row; "
                "32 rows T=0.8, 16 rows top_p=0.9 top_k=50 T=1, 16 greedy; ids only")
    return batch.name


def algorithmic_bytes(batch, want_probs: bool) -> int:
    """Bytes the step must move at least once: logits read once (forks share their row),
    per-row parameters and history read once, outputs written once."""
    out = batch.n_rows * 4 * 2  # tokens + status
    if want_probs:
        out += 8 * batch.n_rows * batch.vocab
    return batch.unique_logit_bytes() + batch.param_bytes() + batch.history_bytes() + out


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(workload: str):
    """dram bytes per launch of the dominant kernel, from the committed ncu summaries
    (profiles/*.md lines `kernel_hash: ...`, `workload: ...` and
    `dram_bytes_per_launch: ...`), if one was taken on this workload with the
    kernels as they are now."""
    pdir = os.path.join(ROOT, "profiles")
    want = kernel_hash()
    try:
        names = sorted(os.listdir(pdir))
    except OSError:
        return None
    for name in names:
        if not name.endswith(".md"):
            continue
        fields = {}
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                if ":" in line and not line.startswith(("|", "#", " ")):
                    k, _, v = line.partition(":")
                    fields[k.strip()] = v.strip()
        if fields.get("workload", workload) != workload:
            continue
        if fields.get("kernel_hash") == want and "dram_bytes_per_launch" in fields:
            try:
                return {"dram_bytes_per_launch": int(fields["dram_bytes_per_launch"]), "source": name}
            except ValueError:
                continue
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={interval_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.lines = []
        if self.proc:
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or [l for (_, l) in self.lines]
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in rows:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[2:6]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, device) -> float:
    """The slowest replica's time (the job ends with the last one); every rank gets
    it. Needs an initialised process group; ends with a barrier."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_rows_per_second(world: int, n_rows: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every replica samples `n_rows` rows per step."""
    return world * n_rows * steps / (ms / 1e3)


def oracle_rows_per_second(batch, seconds: float, nthreads: int):
    """Time the CPU oracle on whole batches (rotating rows) for about `seconds`."""
    import oracle

    n = batch.n_rows
    t0 = time.perf_counter()
    done = 0
    chunk = max(1, min(n, nthreads))
    start = 0
    while True:
        rows = [(start + i) % n for i in range(chunk)]
        oracle.sample(batch, rows=rows, want_probs=batch.want_probs, nthreads=nthreads)
        done += chunk
        start = (start + chunk) % n
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


def run_reference(args):
    """The CPU oracle as it stands, one row of the batch per step (rotating), one thread."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle

    batch = workloads.make(args.workload)
    oracle.build()
    n = batch.n_rows
    for w in range(args.warmup):
        oracle.sample(batch, rows=[w % n], want_probs=batch.want_probs, nthreads=1)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.sample(batch, rows=[s % n], want_probs=batch.want_probs, nthreads=1)
    el = time.perf_counter() - t0
    value = args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * n / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": describe(batch), "n_rows": n,
                                        "vocab": batch.vocab},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"one row of the {n}-row batch per step, rotating; "
                                   f"{args.steps} rows in {el:.1f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import decode_step_token_gb300 as pkg
    from decode_step_token_gb300 import build as libbuild
    from workloads import device as wdev

    libbuild.build_library()
    batch = workloads.make(args.workload)
    want = batch.want_probs
    step_bytes = algorithmic_bytes(batch, want)
    in_bytes = batch.n_logit_rows * batch.row_stride * batch.elem_bytes
    copies = max(2, int(np.ceil(3 * L2_BYTES / max(1, in_bytes)))) if not args.no_rotate else 1
    copies = min(copies, 64)
    sampler = pkg.Sampler(max_rows=batch.n_rows, max_vocab=batch.vocab, device=local)
    d = wdev.to_device(batch, dev, want, copies=copies)
    arg_blocks = [wdev.sample_args(sampler, batch, d, copy_index=i) for i in range(copies)]

    stream = torch.cuda.Stream(device=dev)
    sampler.stat(0, reset=True)
    with torch.cuda.stream(stream):
        for i in range(copies):  # first launches outside capture set kernel attributes
            sampler.sample_args(arg_blocks[i], stream.cuda_stream)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(copies):
                sampler.sample_args(arg_blocks[i], torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize(dev)

    reps_w = max(1, int(np.ceil(args.warmup / copies)))
    reps = max(1, int(np.ceil(args.steps / copies)))
    steps = reps * copies
    with torch.cuda.stream(stream):
        for _ in range(reps_w):
            graph.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = ClockSampler(local) if not args.no_clocks else None
    time.sleep(0.1 if clocks else 0)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop(t0, t1) if clocks else None
    if world > 1:
        ms = max_over_ranks(ms, dev)
    ms_step = ms / steps
    value = job_rows_per_second(world, batch.n_rows, steps, ms)

    exact_rows = sampler.stat(0, reset=True)
    if rank != 0:
        return
    tokens = d["out_tokens"].cpu().numpy()

    # e2e through the host-buffer entry point
    e2e = run_e2e(pkg, batch, local, args.e2e_steps) if not args.no_e2e else None

    peak, peak_kind = measured_peaks()
    launch_s = ms_step / 1e3
    achieved = step_bytes / launch_s / 1e9
    tr = traffic_record(batch.name)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": tr["dram_bytes_per_launch"] if tr else None,
            "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth), kernel timed inside a graph "
                           f"of back-to-back launches",
            "algorithmic_bytes_per_launch": step_bytes}
    cpu = None
    if not args.no_cpu:
        cores = os.cpu_count() or 1
        rps, nrows, el = oracle_rows_per_second(batch, args.cpu_seconds, cores)
        cpu = {"value": rps, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{nrows} rows of the same batch ({el:.1f} s, {cores} threads)"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": reps_w * copies, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": describe(batch), "n_rows": batch.n_rows, "vocab": batch.vocab,
                   "logits_dtype": batch.dtype, "l2": f"rotating {copies} input copies "
                   f"({copies * in_bytes / 1e6:.0f} MB > L2)", "replicas": world},
        "us_per_step": ms_step * 1e3,
        "hbm_gbs": achieved,
        "tokens_per_s": value,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": steps,
        "exact_path_rows_per_step": exact_rows / (steps + (reps_w + 1) * copies),
        "clocks": clk,
        "kernel_hash": kernel_hash(),
        "first_tokens": tokens[:8].tolist(),
    }
    print(json.dumps(line), flush=True)
    sampler.close()


def run_e2e(pkg, batch, device, steps):
    """Rows/s through sampler_sample_host: pinned host inputs copied in, tokens copied
    back, stream synchronised, every step."""
    import torch

    s = pkg.Sampler(max_rows=batch.n_rows, max_vocab=batch.vocab, device=device,
                    max_history=int(batch.hist_ids.size) if batch.hist_ids is not None else 0,
                    host_staging=True)
    keep = []

    def pin(a):
        if a is None:
            return None
        arr = np.ascontiguousarray(a)
        t = torch.from_numpy(arr.view(np.uint8).reshape(-1).copy()).pin_memory()
        keep.append(t)
        return t.data_ptr()

    N, V = batch.n_rows, batch.vocab
    tok = torch.zeros(N, dtype=torch.int32).pin_memory()
    st = torch.zeros(N, dtype=torch.int32).pin_memory()
    pr = torch.zeros((N, V), dtype=torch.float32).pin_memory() if batch.want_probs else None
    lp = torch.zeros((N, V), dtype=torch.float32).pin_memory() if batch.want_probs else None
    args = pkg.sampler_args_t(
        pin(batch.logits), 1 if batch.dtype == "bf16" else 0, N, V, batch.row_stride,
        batch.n_logit_rows, pin(batch.logit_row), pin(batch.temperature), pin(batch.top_k),
        pin(batch.top_p), pin(batch.min_p), pin(batch.presence), pin(batch.frequency),
        pin(batch.repetition), pin(batch.seed), pin(batch.has_seed), pin(batch.stream_id),
        pin(batch.hist_offsets), pin(batch.hist_ids), batch.global_seed, batch.philox_offset,
        None, tok.data_ptr(), pr.data_ptr() if pr is not None else None,
        lp.data_ptr() if lp is not None else None, st.data_ptr())
    stream = torch.cuda.Stream(device=device)
    for _ in range(3):
        s.sample_host_args(args, stream.cuda_stream)
    t0 = time.perf_counter()
    for _ in range(steps):
        s.sample_host_args(args, stream.cuda_stream)
    el = time.perf_counter() - t0
    h2d = (batch.n_logit_rows * V * batch.elem_bytes + batch.param_bytes() + batch.history_bytes())
    d2h = N * 8 + (8 * N * V if batch.want_probs else 0)
    s.close()
    return {"value": N * steps / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-rotate", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
