#!/usr/bin/env python
"""Benchmark of the per-decode-step token sampler.

One step = one sampling call over the whole batch (load, penalties,
temperature, top-k/top-p, min-p, pick, optional probs/logprobs). Default
workload: N=64 rows, V=128000 bf16 logits ~ 2*N(0,1) with one +12 spike per
row; 32 rows T=0.8, 16 rows top_p=0.9 + top_k=50, 16 greedy; token ids only.

Prints one JSON line (rank 0). Our arm: exactly --steps steps, replayed from
CUDA graphs over rotating input copies larger than L2, one CUDA-event pair per
replay on the launching stream; the per-step distribution (median, IQR) comes
from those replays, and from a sustained run of at least half a second when
the requested steps take less. `e2e` goes through the host-buffer C entry
point; `roofline` is for the sampling kernel; `cpu_baseline` = the CPU oracle
on a bounded sample at one thread and at every core; `ablation` times the
per-family workloads (plain -> +top-k/top-p -> +min-p -> +penalties);
`logprob_outputs` times the same step with the per-row logprob outputs
(sampled token + top 5, scaled and unscaled); `extensions` with a
vocabulary mask, with logit_bias lists, with a min_tokens ban and with NaN
sanitising; `lm_head` the LM-head GEMM (tcgen05) before the sampler, alone,
chained, and against cuBLAS.
`--impl reference` times the CPU oracle itself (the only reference this
sampler has), one row per step. Several GPUs run independent replicas (rows
are independent: no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
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
SUSTAINED_S = 0.5


# the device code of the kernel a workload runs: the kernel the roofline and the
# committed ncu counters are about (the host-side headers the kernels also
# include declare other kernels' entry points too)
KERNEL_SOURCES = {
    "slice": ("slice_kernel.cu", "slice_kernel_ext.cu", "slice_kernel.cuh", "slice_sampler.cuh",
              "row_sampler.cuh", "philox.cuh", "ptx.cuh"),
    "group": ("group_kernel.cu", "group_sampler.cuh", "group_sampler_kernel.cuh", "row_sampler.cuh",
              "philox.cuh", "ptx.cuh"),
}


def kernel_kind(batch) -> str:
    """Which kernel the library runs a batch on: the small-batch (slice) kernel for
    at most 256 rows without history or materialised outputs, else the fork-group
    kernel."""
    slice_ok = batch.n_rows <= 256 and batch.hist_offsets is None and not batch.want_probs
    return "slice" if slice_ok else "group"


def kernel_hash(kind: str = "slice") -> str:
    """Hash of the device sources of one kernel."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
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


def traffic_record(workload: str, kind: str = "slice"):
    """dram bytes per launch of the sampling kernel, from the committed ncu summaries
    (profiles/*.md lines `kernel_hash: ...`, `workload: ...` and
    `dram_bytes_per_launch: ...`), if one was taken on this workload with the
    kernels as they are now."""
    pdir = os.path.join(ROOT, "profiles")
    want = kernel_hash(kind)
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


def cpu_info():
    """CPU model and logical core count (lscpu, else /proc/cpuinfo)."""
    model, cores = None, os.cpu_count() or 1
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and not model:
                model = v.strip()
            if k.strip() == "CPU(s)":
                try:
                    cores = int(v.strip())
                except ValueError:
                    pass
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.partition(":")[2].strip()
                        break
        except OSError:
            pass
    return {"model": model or "unknown", "logical_cpus": cores}


def stats_us(per_step_us):
    """median / IQR / p10 / p90 of per-step microseconds."""
    a = np.asarray(per_step_us, dtype=np.float64)
    if a.size == 0:
        return None
    q = np.percentile(a, [10, 25, 50, 75, 90])
    return {"median_us": float(q[2]), "iqr_us": [float(q[1]), float(q[3])], "p10_us": float(q[0]),
            "p90_us": float(q[4]), "mean_us": float(a.mean()), "samples": int(a.size)}


class ClockSampler:
    """nvidia-smi clock / throttle samples while a timed region runs."""

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

    def window(self, t0, t1):
        """Summary of the samples taken between t0 and t1 (perf_counter), or None."""
        rows = [l for (t, l) in self.lines if t0 <= t <= t1]
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

    def stop(self):
        if not self.proc:
            return
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()


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
    """Time the CPU oracle on whole chunks of rows (rotating) for about `seconds`."""
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
    """The CPU oracle as it stands, one thread; a step is one row of the batch
    (rotating), so that the whole run stays short."""
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
    cpu = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": describe(batch), "n_rows": n, "vocab": batch.vocab,
                   "step": f"one row of the {n}-row batch (rotating); rows/s = steps / time"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "cpu_model": cpu["model"],
                         "sample": f"{args.steps} rows of the {n}-row batch, one per step, "
                                   f"rotating; {el:.2f} s at one thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Replayer:
    """CUDA graphs of sampling calls over rotating input copies: `full` holds one
    call per copy; `part(r)` the first r copies (for a step count that is not a
    multiple of the copies). Each replay is bracketed by its own event pair."""

    def __init__(self, torch, sampler, arg_blocks, stream):
        self.torch = torch
        self.sampler = sampler
        self.args = arg_blocks
        self.stream = stream
        self.R = len(arg_blocks)
        self.graphs = {}

    def graph(self, r):
        if r not in self.graphs:
            torch = self.torch
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(r):
                        self.sampler.sample_args(self.args[i], torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            self.graphs[r] = g
        return self.graphs[r]

    def run(self, steps):
        """Replay exactly `steps` calls; returns (total ms, [(calls, ms) per replay])."""
        torch = self.torch
        plan = [self.R] * (steps // self.R) + ([steps % self.R] if steps % self.R else [])
        for r in set(plan):
            self.graph(r)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(plan) + 1)]
        with torch.cuda.stream(self.stream):
            ev[0].record(self.stream)
            for i, r in enumerate(plan):
                self.graphs[r].replay()
                ev[i + 1].record(self.stream)
        torch.cuda.synchronize()
        per = [(r, ev[i].elapsed_time(ev[i + 1])) for i, r in enumerate(plan)]
        return ev[0].elapsed_time(ev[-1]), per


def per_step_us(per):
    return [1e3 * ms / r for (r, ms) in per]


def prepare(torch, pkg, wdev, batch, dev, local, no_rotate=False):
    in_bytes = batch.n_logit_rows * batch.row_stride * batch.elem_bytes
    copies = 1 if no_rotate else min(64, max(2, int(np.ceil(3 * L2_BYTES / max(1, in_bytes)))))
    hist = int(batch.hist_ids.size) if batch.hist_ids is not None else 0
    sampler = pkg.Sampler(max_rows=batch.n_rows, max_vocab=batch.vocab, device=local, max_history=hist)
    d = wdev.to_device(batch, dev, batch.want_probs, copies=copies)
    arg_blocks = [wdev.sample_args(sampler, batch, d, copy_index=i) for i in range(copies)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(copies):  # the first calls, outside capture, set kernel attributes
            sampler.sample_args(arg_blocks[i], stream.cuda_stream)
    torch.cuda.synchronize(dev)
    return sampler, d, Replayer(torch, sampler, arg_blocks, stream), copies, in_bytes


def sustained(rep, seconds):
    """Whole replays for at least `seconds`; per-step microseconds of each replay."""
    out, t_end = [], time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        _, per = rep.run(rep.R * max(1, int(np.ceil(2000 / rep.R))))
        out.extend(per_step_us(per))
    return out


def host_call_us(sampler, arg_blocks, stream, n=200):
    """CPU time of one sampling call through the binding (enqueue only, no sync)."""
    import torch

    ts = []
    for i in range(n):
        t0 = time.perf_counter()
        sampler.sample_args(arg_blocks[i % len(arg_blocks)], stream.cuda_stream)
        ts.append(1e6 * (time.perf_counter() - t0))
        if i % 32 == 31:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return stats_us(ts)


class LogprobReplayer(Replayer):
    """Replays of sampler_sample_ex calls (logprob outputs or another extension)."""

    def __init__(self, torch, sampler, arg_blocks, stream, lp_kw):
        super().__init__(torch, sampler, arg_blocks, stream)
        self.lp_kw = lp_kw

    def graph(self, r):
        if r not in self.graphs:
            torch = self.torch
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(r):
                        self.sampler.sample_ex_args(self.args[i], stream=torch.cuda.current_stream().cuda_stream,
                                                          **self.lp_kw)
            torch.cuda.synchronize()
            self.graphs[r] = g
        return self.graphs[r]


def run_logprob_outputs(torch, sampler, rep, batch, dev, top_n, seconds):
    """Median step time with the per-row logprob outputs (sampled token + top_n),
    scaled and unscaled, on the same rotating inputs."""
    N = batch.n_rows
    out = {"top_n": top_n, "output_bytes_per_step": N * 4 + N * top_n * 8,
           "materialised_bytes_per_step": 8 * N * batch.vocab}
    for unscaled in (False, True):
        kw = dict(top_n=top_n, unscaled=unscaled,
                  out_token_logprob=torch.empty(N, dtype=torch.float32, device=dev),
                  out_top_ids=torch.empty((N, top_n), dtype=torch.int32, device=dev),
                  out_top_logprobs=torch.empty((N, top_n), dtype=torch.float32, device=dev))
        lr = LogprobReplayer(torch, sampler, rep.args, rep.stream, kw)
        with torch.cuda.stream(rep.stream):
            for a in rep.args:
                sampler.sample_ex_args(a, stream=rep.stream.cuda_stream, **kw)
        torch.cuda.synchronize()
        lr.run(lr.R * 2)
        out["unscaled" if unscaled else "scaled"] = stats_us(sustained(lr, seconds))
    return out


def run_extensions(torch, pkg, wdev, batch, dev, local, seconds):
    """Median step time of the same batch with each sampler_sample_ex extension:
    a grammar-style vocabulary mask (about 10 % of tokens allowed per row), 64
    logit_bias entries per row, 16 stop tokens banned on every row (min_tokens),
    and NaN sanitising over the same logits and over logits with 0.1 % NaN."""
    out = {}
    n, V = batch.n_rows, batch.vocab
    words = (V + 31) // 32
    mask = workloads.vocab_mask(7, n, V, allowed=0.1, full_rows=0)
    offs = np.arange(0, 64 * n + 1, 64, dtype=np.int32)
    rng = np.random.Generator(np.random.PCG64(8))
    ids = rng.integers(0, V, size=int(offs[-1])).astype(np.int32)
    vals = (rng.standard_normal(ids.size) * 5).astype(np.float32)
    left = np.ones(n, np.int32)
    soffs = np.arange(0, 16 * n + 1, 16, dtype=np.int32)
    sids = rng.integers(0, V, size=16 * n).astype(np.int32)
    x = batch.logits.copy()
    at = rng.random(x.shape) < 0.001
    x[at] = np.uint16(0x7FC0) if batch.dtype == "bf16" else np.float32(np.nan)
    cases = (("vocab_mask_10pct", dict(vocab_mask=mask), n * words * 4),
             ("logit_bias_64", dict(bias_offsets=offs, bias_ids=ids, bias_values=vals),
              offs.nbytes + ids.nbytes + vals.nbytes),
             ("min_tokens_16_stops", dict(min_tokens_left=left, stop_offsets=soffs, stop_ids=sids),
              left.nbytes + soffs.nbytes + sids.nbytes),
             ("sanitize_nan_no_nan", dict(sanitize_nan=True), 0),
             ("sanitize_nan_0.1pct", dict(logits=x, sanitize_nan=True), 0))
    for name, kw, extra in cases:
        b = batch.with_(**kw)
        s, d, rep, copies, _ = prepare(torch, pkg, wdev, b, dev, local)
        lr = LogprobReplayer(torch, s, rep.args, rep.stream, wdev.ext_kw(d))
        with torch.cuda.stream(rep.stream):
            for a in rep.args:
                s.sample_ex_args(a, stream=rep.stream.cuda_stream, **wdev.ext_kw(d))
        torch.cuda.synchronize()
        lr.run(lr.R * 2)
        st = stats_us(sustained(lr, seconds))
        st["extra_bytes_per_step"] = int(extra)
        st["exact_path_rows"] = s.stat(0, reset=True)
        out[name] = st
        s.close()
        del d, rep, lr
        torch.cuda.empty_cache()
    return out


class FnReplayer(Replayer):
    """CUDA graphs of R calls of fn(stream) (same run() / sustained() interface)."""

    def __init__(self, torch, fn, stream, R):
        super().__init__(torch, None, [None] * R, stream)
        self.fn = fn

    def graph(self, r):
        if r not in self.graphs:
            torch = self.torch
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g, stream=self.stream):
                    for _ in range(r):
                        self.fn(torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            self.graphs[r] = g
        return self.graphs[r]


def run_lm_head(torch, pkg, wdev, dev, local, seconds, n=64, V=128000, K=4096):
    """The LM-head step: logits = hidden x weight^T (bf16, K = 4096, weight 1 GB,
    larger than L2) on the tcgen05 GEMM, then the mixed batch's sampling on
    them. Times the GEMM alone, the sampler alone on its logits (L2-warm), the
    two in plain stream order, the two chained by sampler_lm_head_sample
    (programmatic dependent launch), cuBLAS (torch.matmul) alone and followed
    by the sampler."""
    import workloads

    hidden_bits, _, b = workloads.lm_head(6, n, V, K, weight=False)
    gen = torch.Generator(device=dev).manual_seed(6)
    w = (torch.randn((V, K), generator=gen, device=dev) * (2.0 / np.sqrt(K))).to(torch.bfloat16)
    torch.cuda.empty_cache()
    h = torch.from_numpy(hidden_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    sampler = pkg.Sampler(max_rows=n, max_vocab=V, device=local)
    d = wdev.to_device(b, dev, False)
    args = wdev.sample_args(sampler, b, d)
    logits = d["logits"][0]
    stream = torch.cuda.Stream(device=dev)
    variants = {
        "gemm": lambda st: sampler.lm_head(h, w, logits, stream=st),
        "sampler": lambda st: sampler.sample_args(args, st),
        "chained": lambda st: sampler.lm_head_sample_args(args, h, w, stream=st),
        "cublas_gemm": lambda st: torch.matmul(h, w.t(), out=logits),
    }
    variants["gemm_then_sampler"] = lambda st: (variants["gemm"](st), variants["sampler"](st))
    variants["cublas_then_sampler"] = lambda st: (variants["cublas_gemm"](st), variants["sampler"](st))
    out = {"n_rows": n, "vocab": V, "hidden_dim": K}
    with torch.cuda.stream(stream):
        for f in variants.values():  # first calls outside capture (kernel attributes, cuBLAS handles)
            f(stream.cuda_stream)
    torch.cuda.synchronize()
    for name, f in variants.items():
        rep = FnReplayer(torch, f, stream, 8)
        rep.run(16)
        out[name] = stats_us(sustained(rep, seconds))
    gemm_bytes = V * K * 2 + n * K * 2 + n * V * 2
    peak, kind = measured_peaks()
    t = out["gemm"]["median_us"] * 1e-6
    out["gemm_roofline"] = {"bound": "hbm", "algorithmic_bytes": gemm_bytes, "achieved": gemm_bytes / t / 1e9,
                            "peak": peak, "unit": "GB/s", "frac": gemm_bytes / t / 1e9 / peak,
                            "peak_source": f"{kind} hbm_gbs", "tflops": 2.0 * n * V * K / t / 1e12}
    # what the programmatic dependent launch saves against the same two kernels in
    # plain stream order (the sampler alone re-reads logits that stay in L2)
    out["chained_saving_us"] = out["gemm_then_sampler"]["median_us"] - out["chained"]["median_us"]
    out["timeouts"] = sampler.stat(1)
    sampler.close()
    del w, h, d
    torch.cuda.empty_cache()
    return out


def run_ablation(torch, pkg, wdev, dev, local, seconds):
    """Median step time of each per-family workload (plain -> +top-k/top-p ->
    +min-p -> +penalties) at N=64, V=128000 bf16."""
    res = {}
    for stage in workloads.ABLATION_STAGES:
        b = workloads.ablation(stage)
        s, d, rep, copies, _ = prepare(torch, pkg, wdev, b, dev, local)
        rep.run(copies * 2)
        st = stats_us(sustained(rep, seconds))
        st["algorithmic_bytes"] = algorithmic_bytes(b, b.want_probs)
        st["exact_path_rows"] = s.stat(0, reset=True)
        res[stage] = st
        s.close()
        del d, rep
        torch.cuda.empty_cache()
    return res


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
    step_bytes = algorithmic_bytes(batch, batch.want_probs)
    sampler, d, rep, copies, in_bytes = prepare(torch, pkg, wdev, batch, dev, local, args.no_rotate)
    sampler.stat(0, reset=True)

    # warm-up: exactly --warmup calls (at least 3), untimed
    rep.run(max(3, args.warmup))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = ClockSampler(local) if not args.no_clocks else None
    time.sleep(0.1 if clocks else 0)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    ms, per = rep.run(args.steps)
    t1 = time.perf_counter()
    clk = clocks.window(t0, t1) if clocks else None
    if world > 1:
        ms = max_over_ranks(ms, dev)
    ms_step = ms / args.steps
    value = job_rows_per_second(world, batch.n_rows, args.steps, ms)
    exact_rows = sampler.stat(0, reset=True)

    # the per-step distribution: the timed replays themselves when they last long
    # enough, else a sustained run of whole replays (clocks sampled there too)
    dist_src = "the timed region's replays"
    samples = per_step_us(per)
    sus_clk = None
    if ms / 1e3 < SUSTAINED_S or len(samples) < 20:
        s0 = time.perf_counter()
        samples = sustained(rep, SUSTAINED_S)
        s1 = time.perf_counter()
        sus_clk = clocks.window(s0, s1) if clocks else None
        dist_src = f"a sustained run of whole {copies}-call replays ({s1 - s0:.2f} s)"
    if clocks:
        clocks.stop()
    if clk is None or clk.get("samples", 0) < 3:
        clk = dict(sus_clk or clk or {}, window="sustained run (the timed region was too short to sample)") \
            if (sus_clk or clk) else None
    timing = stats_us(samples)
    timing["source"] = dist_src
    timing["timed_region_s"] = ms / 1e3

    if rank != 0:
        return
    tokens = d["out_tokens"].cpu().numpy()
    host = host_call_us(sampler, rep.args, rep.stream)

    e2e = run_e2e(pkg, batch, local, args.e2e_steps) if not args.no_e2e else None

    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (ms_step / 1e3) / 1e9
    tr = traffic_record(batch.name, kernel_kind(batch))
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": tr["dram_bytes_per_launch"] if tr else None,
            "traffic_source": (f"ncu capture summarised in profiles/{tr['source']} (same kernel "
                               f"sources), not measured in this run") if tr else None,
            "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth), of {peak_kind}",
            "algorithmic_bytes_per_launch": step_bytes,
            "launch_time": "mean of the timed region (CUDA events, graph replays)"}
    cpu = None
    if not args.no_cpu:
        info = cpu_info()
        cores = info["logical_cpus"]
        rps, nrows, el = oracle_rows_per_second(batch, args.cpu_seconds, cores)
        rps1, nrows1, el1 = oracle_rows_per_second(batch, args.cpu_seconds / 2, 1)
        cpu = {"value": rps, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": info["model"],
               "sample": f"{nrows} rows of the same batch ({el:.1f} s, {cores} threads)",
               "one_thread": {"value": rps1, "unit": UNIT, "sample": f"{nrows1} rows ({el1:.1f} s)"}}
    abl = None
    lpo = None
    ext = None
    lmh = None
    if not args.no_ablation and args.workload == "mixed":
        lpo = run_logprob_outputs(torch, sampler, rep, batch, dev, 5, args.ablation_seconds)
        ext = run_extensions(torch, pkg, wdev, batch, dev, local, args.ablation_seconds)
        abl = run_ablation(torch, pkg, wdev, dev, local, args.ablation_seconds)
        lmh = run_lm_head(torch, pkg, wdev, dev, local, args.ablation_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": describe(batch), "n_rows": batch.n_rows, "vocab": batch.vocab,
                   "logits_dtype": batch.dtype, "compute": "fp32 (exact ties settled in fp64)",
                   "l2": f"rotating {copies} input copies ({copies * in_bytes / 1e6:.0f} MB > L2)",
                   "replicas": world},
        "us_per_step": ms_step * 1e3,
        "timing": timing,
        "host_call_us": host,
        "hbm_gbs": achieved,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "exact_path_rows_per_step": exact_rows / args.steps,
        "clocks": clk,
        "ablation": abl,
        "logprob_outputs": lpo,
        "extensions": ext,
        "lm_head": lmh,
        "kernel_hash": kernel_hash(kernel_kind(batch)),
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
    ts = []
    t0 = time.perf_counter()
    for _ in range(steps):
        a = time.perf_counter()
        s.sample_host_args(args, stream.cuda_stream)
        ts.append(1e6 * (time.perf_counter() - a))
    el = time.perf_counter() - t0
    h2d = (batch.n_logit_rows * V * batch.elem_bytes + batch.param_bytes() + batch.history_bytes())
    d2h = N * 8 + (8 * N * V if batch.want_probs else 0)
    s.close()
    return {"value": N * steps / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "per_call": stats_us(ts)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ablation-seconds", type=float, default=0.3)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-rotate", action="store_true")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--lm-head-only", action="store_true",
                    help="run only the LM-head leg (GEMM, sampler, chained, cuBLAS) and print its JSON")
    ap.add_argument("--hidden-dim", type=int, default=4096, help="K of the LM-head leg")
    args = ap.parse_args()
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.lm_head_only:
        import torch

        import decode_step_token_gb300 as pkg
        from workloads import device as wdev

        print(json.dumps(run_lm_head(torch, pkg, wdev, "cuda:0", 0, args.ablation_seconds, K=args.hidden_dim)),
              flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
