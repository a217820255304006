#!/usr/bin/env python3
"""Benchmark of the NVFP4 block-scaled batched GEMV on GB300.

One step is one GEMV call (the whole path: stream A and its block scales, stage the vector,
decode, scale, reduce, fp16 store) over one batch of seeded synthetic input.  The default workload
is the decode GEMV M=7168, K=16384, L=1 (66.1 MB per call).  Prints ONE JSON line:

  metric / value / unit   achieved HBM GB/s of algorithmic bytes (M*K*L/2 + M*K*L/16 + K*L/2 +
                          K*L/16 + 2*M*L per call), whole job over all ranks, inputs resident in HBM
  us_per_call, pct_of_peak
  per_config              the five decode workloads c1..c5 in the same run: us per call over the
                          K timed steps and in steady state (graphs of 1000 calls), GB/s, fraction
                          of peak, strict stream order, the plan
  small_ml                few output rows (M*L = 16..512) with long K: the split-K regime
  e2e                     the same metric through the public call with host buffers: every step
                          copies its inputs from pinned host memory and reads back c
  roofline                dominant kernel vs the measured HBM copy bandwidth
  cpu_baseline            the plain C oracle (fp64) on the host cores, one thread and OpenMP
  clocks                  nvidia-smi samples taken during the timed region

Timing: W warm-up steps, then exactly K steps timed with CUDA events on the launching stream,
barrier + synchronize on both sides, max over ranks.  L2 residency is defeated by rotating over
copies of the inputs totalling more than 3x the L2 size (each step reads a different copy).  The
launches are captured in CUDA graphs (up to 1000 calls per graph), and a short spin kernel runs
ahead of the start event, so that by the time the device reaches the start event the host has
queued the timed graphs: the device-timed region holds the K calls, not the host's launch latency.

Multi-GPU: the GEMV needs no exchange between GPUs, so each rank runs an independent replica on
its own GPU (weak scaling) and rank 0 reports the sum of bytes over the max time.  Under torchrun
(WORLD_SIZE set) --gpus must equal WORLD_SIZE; without it, --gpus N > 1 starts the N ranks itself.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c2] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "NVFP4 batched GEMV achieved HBM GB/s (% of GB300 peak) and us/call per MxKxL"
GRAPH_CHUNK = 1000
FLAG_EARLY_WEIGHTS = 1      # nvfp4_plan.flags: A and sfa are not written by preceding work
FLAG_QUANTIZE_IN_GEMV = 4   # nvfp4_plan.flags: quantize the bf16 vector inside the GEMV kernel
FLAG_NO_L2_PREFETCH = 16    # nvfp4_plan.flags: strict order without the L2 prefetch before the wait
KERNEL_NAMES = {1: "gemv_simple_kernel", 2: "gemv_stream_kernel", 3: "gemv_tma_kernel",
                4: "gemv_tma_rv_kernel", 5: "gemv_tc_kernel", 6: "gemv_shift_kernel"}
DEFAULT_PEAK_GBS = 6800.0   # only if MEASURED_PEAKS.json is absent
PREROLL_CYCLES = 200_000    # spin kernel ahead of every start event (~0.1 ms at 2 GHz)
NOMINAL_HBM_GBS = 7900.0    # GB300's nominal HBM3e rate, reported beside the measured-peak fraction


# ---------------------------------------------------------------------------- distributed helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_ranks(n: int, argv) -> int:
    """Starts bench.py once per rank (RANK / LOCAL_RANK / WORLD_SIZE / MASTER_* set, as torchrun
    would) and waits for all of them; returns the worst exit code."""
    port = str(free_port())
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv], env=env))
    codes = [p.wait() for p in procs]
    return max(abs(c) for c in codes)


def dist_init(world):
    if world <= 1:
        return None
    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_scalar(dist, x: float, op: str) -> float:
    """max / sum of a host scalar over ranks (gloo; no data-path collective)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(dist, bytes_per_rank: float, seconds: float):
    """Whole-job throughput: bytes summed over ranks / slowest rank's time."""
    total = reduce_scalar(dist, bytes_per_rank, "sum")
    slowest = reduce_scalar(dist, seconds, "max")
    return total, slowest


# ---------------------------------------------------------------------------- peaks, clocks

def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return DEFAULT_PEAK_GBS, "fallback"


CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling (200 ms) of one GPU while the timed region runs."""

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def query_once(self):
        try:
            out = subprocess.run(["nvidia-smi", "-i", self.gpu_id, "--format=csv,noheader,nounits",
                                  "--query-gpu=" + ",".join(CLOCK_FIELDS)],
                                 capture_output=True, text=True, timeout=20)
            return [ln for ln in out.stdout.splitlines() if ln.strip()]
        except (OSError, subprocess.SubprocessError):
            return []

    def __enter__(self):
        self.before = self.query_once()
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--format=csv,noheader,nounits", "-lms", "200",
                 "--query-gpu=" + ",".join(CLOCK_FIELDS)], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
        self.after = self.query_once()
        return False

    def summary(self):
        lines = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                lines = [ln for ln in f.read().splitlines() if ln.strip()]
            os.unlink(self.path)
        rows = [r.split(", ") for r in (lines or (self.before + self.after))]
        rows = [r for r in rows if len(r) == len(CLOCK_FIELDS)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------- traffic record

# The headers the register-vector TMA kernel (the kernel the roofline line reports) is built from.
RV_KERNEL_HEADERS = ("gemv_kernels.cuh", "gemv_tma.cuh", "nvfp4_device.cuh", "quantize.cuh")


def _code_only(text: str) -> str:
    """C++ source with comments removed and whitespace collapsed (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest() -> str:
    """Digest of the code (comments and layout excluded) of the device headers the reported kernel
    is built from; the host planner and the other kernels' headers are not part of it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_nvfp4_gemv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f in RV_KERNEL_HEADERS:
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on these sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload_name}.txt")
    try:
        kv = {}
        with open(path) as f:
            for ln in f:
                if "=" in ln and not ln.lstrip().startswith("#"):
                    k, v = ln.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sources_sha256_16") != kernel_source_digest():
            return None
        return float(kv["dram_bytes_read_per_launch"]) + float(kv["dram_bytes_write_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def headline_workload(args):
    """The timed workload and its name: a named decode config, or any M x K x L (--shape) drawn
    like c5 (uniform packed bytes, block scales of powers of two from 2^-3 to 2^2)."""
    if not args.shape:
        return workloads.make(args.config), args.config
    M, K, L = parse_shape(args.shape)
    name = f"{M}x{K}x{L}"
    return workloads.random_workload(M, K, L, seed=M + K + L,
                                     scale_bytes=workloads.pow2_scale_bytes(-3, 2), g_a=0.5,
                                     g_b=1.0, name=name), name


def parse_shape(text):
    """'MxKxL' (or 'MxK', L = 1) -> (M, K, L); K a positive multiple of 16."""
    parts = [int(v) for v in text.lower().split("x")]
    if len(parts) == 2:
        parts.append(1)
    if len(parts) != 3 or min(parts) < 1 or parts[1] % 16:
        raise ValueError(f"--shape wants MxKxL with K a multiple of 16, not {text!r}")
    return tuple(parts)


# ---------------------------------------------------------------------------- our arm

def _device_inputs(w, n_copies, device):
    """n_copies copies of the workload's inputs at distinct addresses: one pool allocation per
    operand (copy i is row i of the pool), filled by one device copy each."""
    import torch

    sets = [{} for _ in range(n_copies)]
    for k in ("A", "sfa", "b", "sfb"):
        x = np.ascontiguousarray(getattr(w, k))
        base = torch.from_numpy(x.reshape(1, -1)).to(device)
        pool = base.expand(n_copies, -1).contiguous()
        for i in range(n_copies):
            sets[i][k] = pool[i].view(x.shape)
    return sets


def _copies_for(bytes_per_call, device):
    """Input copies whose total exceeds 3x the L2 size (at least 2)."""
    import torch

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    return max(2, -(-3 * l2 // bytes_per_call) + 1), l2


def workload_config(w, name, world):
    """The `config` object both arms print: the workload, and how the GPU arm keeps each call's
    inputs out of L2 (rotated copies larger than 3x L2)."""
    import torch

    bytes_call = w.algorithmic_bytes
    if torch.cuda.is_available():
        n_copies, l2 = _copies_for(bytes_call, torch.device("cuda", torch.cuda.current_device()))
        l2_text = (f"GPU arm: inputs rotated over {n_copies} copies "
                   f"({n_copies * bytes_call / 1e6:.0f} MB > 3x L2 {l2 / 1e6:.0f} MB)")
    else:
        l2_text = "GPU arm: inputs rotated over copies larger than 3x L2 (no GPU on this host)"
    return {"workload": f"NVFP4 decode GEMV M={w.M} K={w.K} L={w.L} ({name})",
            "M": w.M, "K": w.K, "L": w.L, "bytes_per_call": bytes_call, "l2": l2_text,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def _preroll():
    """A spin kernel on the current stream ahead of a start event: while it runs, the host queues
    the start event and the timed graphs, so the device-timed region starts with the first call
    rather than with the host's graph launch."""
    import torch

    torch.cuda._sleep(PREROLL_CYCLES)


class GraphTimer:
    """`steps` calls of fn(i) captured in CUDA graphs of up to GRAPH_CHUNK calls (a full graph
    repeated, plus one graph of the remainder), after `warmup` uncaptured calls."""

    def __init__(self, fn, steps, warmup, stream):
        import torch

        self.stream, self.steps = stream, steps
        with torch.cuda.stream(stream):
            for i in range(max(warmup, 1)):          # uncaptured warm-up (caches device info too)
                fn(i)
        stream.synchronize()
        self.chunk = min(GRAPH_CHUNK, steps)
        self.full = self._capture(fn, self.chunk)
        rem = steps % self.chunk
        self.rem = self._capture(fn, rem) if rem else None
        with torch.cuda.stream(stream):              # graph warm-up
            self.full.replay()
        stream.synchronize()

    def _capture(self, fn, count):
        import torch

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(count):
                fn(i)
        return g

    def replay_all(self):
        for _ in range(self.steps // self.chunk):
            self.full.replay()
        if self.rem is not None:
            self.rem.replay()

    def time(self, dist, device, sampler=None):
        """Seconds for the `steps` calls: barrier + synchronize on both sides, the pre-roll spin
        kernel, then CUDA events on the launching stream around the replays."""
        import torch

        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ctx = sampler if sampler is not None else _Null()
        with ctx, torch.cuda.stream(self.stream):
            barrier(dist)
            torch.cuda.synchronize(device)
            _preroll()
            ev0.record(self.stream)
            self.replay_all()
            ev1.record(self.stream)
            torch.cuda.synchronize(device)
            barrier(dist)
        return ev0.elapsed_time(ev1) / 1e3

    def spread(self, device, n_rep=20):
        """p10 / median / p90 of us per call over n_rep replays of the full graph, each between
        two events (after the timed region)."""
        import torch

        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
        with torch.cuda.stream(self.stream):
            _preroll()
            evs[0].record(self.stream)
            for i in range(n_rep):
                self.full.replay()
                evs[i + 1].record(self.stream)
            torch.cuda.synchronize(device)
        per = sorted(evs[i].elapsed_time(evs[i + 1]) * 1e3 / self.chunk for i in range(n_rep))
        return {"replays": n_rep, "calls_per_replay": self.chunk,
                "p10_us": round(per[n_rep // 10], 3), "median_us": round(per[n_rep // 2], 3),
                "p90_us": round(per[(9 * n_rep) // 10], 3)}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def _graph_time(fn, stream, steps, warmup, dist, dev):
    """Seconds and calls for exactly `steps` calls of fn(i) replayed from CUDA graphs."""
    t = GraphTimer(fn, steps, warmup, stream)
    sec = t.time(dist, dev)
    del t
    return sec, steps


def _gemv_caller(pkg, w, sets, outs, plan, stream):
    n = len(sets)

    def call(i):
        s = sets[i % n]
        pkg.nvfp4_gemv_batched_ex(s["A"], s["sfa"], w.g_a, s["b"], s["sfb"], w.g_b, outs[i % n],
                                  w.M, w.K, w.L, stream=stream, plan=plan)
    return call


def plan_with_flags(pkg, M, K, L, plan):
    """The automatic plan a call with these forced fields (flags included) gets on the current
    device: the planner's choice depends on the flags (three CTAs per SM need early weights)."""
    import torch

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    lim = dict(sms=props.multi_processor_count)
    if hasattr(props, "shared_memory_per_block_optin"):
        lim["max_smem_optin"] = props.shared_memory_per_block_optin
    if hasattr(props, "shared_memory_per_multiprocessor"):
        lim["max_smem_sm"] = props.shared_memory_per_multiprocessor
    return pkg.nvfp4_plan_for_limits(M, K, L, plan=plan, **lim).as_dict()


def _plan_name(pkg, w, flags):
    p = plan_with_flags(pkg, w.M, w.K, w.L, {"flags": flags})
    return KERNEL_NAMES.get(p["kernel"], "?"), p


def time_per_config(pkg, device, stream, steps, warmup, dist, names=("c1", "c2", "c3", "c4", "c5"),
                    steady_calls=GRAPH_CHUNK):
    """Every decode workload in the same run.  For each: us per call over `steps` calls (the
    headline's method: early weights, inputs rotated over copies larger than 3x L2), the same
    calls in steady state (graphs of `steady_calls` calls, so the first call's start and the last
    call's drain weigh 1 / steady_calls), and strict stream order (no early weights) over `steps`
    calls.  c1 (18.8 KB) is launch-bound and is listed for completeness."""
    import torch

    peak, _ = measured_peak_gbs()
    out = {}
    for name in names:
        w = workloads.make(name)
        nbytes = w.algorithmic_bytes
        n_copies, _ = _copies_for(nbytes, device)
        sets = _device_inputs(w, n_copies, device)
        outs = [torch.empty((w.L, w.M), dtype=torch.float16, device=device)
                for _ in range(n_copies)]
        row = {"M": w.M, "K": w.K, "L": w.L, "bytes_per_call": nbytes, "copies": n_copies}
        kname, plan = _plan_name(pkg, w, FLAG_EARLY_WEIGHTS)
        row["kernel"], row["plan"] = kname, plan
        for key, flags, n in (("early_weights", FLAG_EARLY_WEIGHTS, steps),
                              ("steady", FLAG_EARLY_WEIGHTS, max(steps, steady_calls)),
                              ("strict_order", 0, steps)):
            t = GraphTimer(_gemv_caller(pkg, w, sets, outs, {"flags": flags}, stream), n, warmup,
                           stream)
            sec = t.time(dist, device)
            tot, slow = aggregate(dist, nbytes * n, sec)
            gbs = tot / slow / 1e9
            row[key] = {"us_per_call": round(sec / n * 1e6, 3), "calls": n,
                        "GB/s": round(gbs, 2), "frac": round(gbs / peak, 4)}
            if flags != FLAG_EARLY_WEIGHTS:
                sp = _plan_name(pkg, w, flags)[1]
                if any(sp[k] != plan[k] for k in sp if k != "flags"):
                    row[key]["plan"] = sp
            del t
        assert not torch.isnan(outs[0]).any().item()
        out[name] = row
        del sets, outs
        torch.cuda.empty_cache()
    out["note"] = ("early_weights: the headline's method over the K timed steps; steady: graphs "
                   f"of {steady_calls} calls; strict_order: no early weights, K steps; frac of "
                   "the measured HBM copy bandwidth")
    return out


def time_small_ml(pkg, device, stream, steps, warmup, dist,
                  shapes=((16, 16384), (64, 16384), (128, 16384), (512, 16384),
                          (16, 65536), (64, 65536), (128, 65536), (512, 65536))):
    """Few output rows with long K (L = 1): the regime where one row per CTA cannot fill the GPU
    and K is split across CTAs.  Each call reads its own copy of A and sfa (a pool of XOR-keyed
    copies larger than 3x L2); the vector is shared.  Graphs of up to 1000 calls."""
    import torch

    peak, _ = measured_peak_gbs()
    out = {}
    for M, K in shapes:
        w = workloads.random_workload(M, K, 1, seed=40 + M + K // 1024,
                                      scale_bytes=workloads.pow2_scale_bytes(-3, 2), g_a=0.5)
        nbytes = w.algorithmic_bytes
        n_copies, _ = _copies_for(M * K * 9 // 16, device)
        A0 = torch.from_numpy(w.A.ravel()).to(device)
        S0 = torch.from_numpy(w.sfa.ravel()).to(device)
        A = torch.empty((n_copies, A0.numel()), dtype=torch.uint8, device=device)
        S = torch.empty((n_copies, S0.numel()), dtype=torch.uint8, device=device)
        for q in range(n_copies):
            torch.bitwise_xor(A0, (29 * q + 3) & 0xFF, out=A[q])
            S[q].copy_(S0)
        b = torch.from_numpy(w.b).to(device)
        sfb = torch.from_numpy(w.sfb).to(device)
        c = torch.empty((n_copies, M), dtype=torch.float16, device=device)
        plan = {"flags": FLAG_EARLY_WEIGHTS}

        def fn(i, A=A, S=S, b=b, sfb=sfb, c=c, n=n_copies, M=M, K=K):
            pkg.nvfp4_gemv_batched_ex(A[i % n], S[i % n], 0.5, b, sfb, 1.0, c[i % n], M, K, 1,
                                      stream=stream, plan=plan)
        n_calls = min(steps, 5000)
        sec, calls = _graph_time(fn, stream, n_calls, warmup, dist, device)
        tot, slow = aggregate(dist, nbytes * calls, sec)
        gbs = tot / slow / 1e9
        kname, p = _plan_name(pkg, w, FLAG_EARLY_WEIGHTS)
        out[f"M={M} K={K}"] = {"us_per_call": round(sec / calls * 1e6, 3), "calls": calls,
                               "GB/s": round(gbs, 2), "frac": round(gbs / peak, 4),
                               "bytes_per_call": nbytes, "kernel": kname, "plan": p}
        del A, S, c
        torch.cuda.empty_cache()
    return out
def time_bf16_vector(pkg, w, sets, outs, stream, steps, warmup, dist):
    """The GEMV with a bf16 activation vector through nvfp4_gemv_batched_bf16, in its two forms:
    the quantizer launched ahead of the GEMV (the default) and the quantization inside the
    register-vector TMA kernel (NVFP4_FLAG_QUANTIZE_IN_GEMV).  Static weights (early-weights flag),
    as in the main timing.  Algorithmic bytes add the bf16 vector read; the packed vector is
    written instead of read (the same bytes)."""
    import torch

    n = len(sets)
    dev = sets[0]["A"].device
    x32 = workloads.normal_bf16(12, "x", w.K * w.L)
    bits = (x32.view(np.uint32) >> 16).astype(np.uint16).view(np.int16).reshape(w.L, w.K)
    gs = float(np.abs(x32).max() / (448.0 * 6.0))
    xs = [torch.from_numpy(bits).to(dev) for _ in range(n)]
    bo = [torch.empty(w.L * w.K // 2, dtype=torch.uint8, device=dev) for _ in range(n)]
    so = [torch.empty(w.L * w.K // 16, dtype=torch.uint8, device=dev) for _ in range(n)]
    bytes_call = w.algorithmic_bytes + 2 * w.K * w.L
    out = {}
    for name, flags in (("quantizer_then_gemv", FLAG_EARLY_WEIGHTS),
                        ("in_gemv", FLAG_EARLY_WEIGHTS | FLAG_QUANTIZE_IN_GEMV)):
        plan = {"flags": flags}

        def fn(i):
            s = sets[i % n]
            pkg.nvfp4_gemv_batched_bf16(s["A"], s["sfa"], w.g_a, xs[i % n], gs, bo[i % n],
                                        so[i % n], outs[i % n], w.M, w.K, w.L, stream=stream,
                                        plan=plan)

        sec, calls = _graph_time(fn, stream, steps, warmup, dist, dev)
        tot, slow = aggregate(dist, bytes_call * calls, sec)
        out[name] = {"us_per_call": round(sec / calls * 1e6, 3), "calls": calls,
                     "GB/s": round(tot / slow / 1e9, 2),
                     "launches_per_call": 1 if flags & FLAG_QUANTIZE_IN_GEMV else 2}
    out["bytes_per_call"] = bytes_call
    out["bytes"] = "A + sfa + bf16 x read + packed x and its scales written + c"
    out["gemv_kernel"] = KERNEL_NAMES.get(pkg.nvfp4_gemv_plan(w.M, w.K, w.L).kernel, "?")
    return out


def time_grouped(pkg, device, stream, steps, warmup, dist, name="g1", n_routes=4):
    """The grouped (mixture-of-experts) decode GEMV on `name`: the experts' weights stay resident
    and every call takes the next of `n_routes` routings (its own offsets and token vectors), as
    decode steps do.  Algorithmic bytes count each expert that owns a token once per call."""
    import torch

    w0 = workloads.make_grouped(name)
    ws = [w0] + [workloads.make_grouped(name, route=r, with_weights=w0) for r in range(1, n_routes)]
    A = torch.from_numpy(w0.A).to(device)
    sfa = torch.from_numpy(w0.sfa).to(device)
    g_a = torch.from_numpy(np.ascontiguousarray(w0.g_a, np.float32)).to(device)
    g_b = torch.from_numpy(np.ascontiguousarray(w0.g_b, np.float32)).to(device)
    per = []
    for w in ws:
        offs = np.cumsum(np.bincount(w.expert_of, minlength=w.E)).astype(np.int32)
        per.append(dict(b=torch.from_numpy(w.b).to(device), sfb=torch.from_numpy(w.sfb).to(device),
                        offs=torch.from_numpy(offs).to(device),
                        c=torch.empty((w.T, w.M), dtype=torch.float16, device=device)))
    M, K, E, T = w0.M, w0.K, w0.E, w0.T

    def call(i):
        r = per[i % n_routes]
        pkg.nvfp4_gemv_grouped(A, sfa, g_a, r["b"], r["sfb"], g_b, r["c"], M, K, E, T,
                               expert_offsets=r["offs"], stream=stream)

    torch.cuda.synchronize(device)
    calls = max(n_routes, steps - steps % n_routes)      # every routing equally often
    sec, calls = _graph_time(call, stream, calls, warmup, dist, device)
    bytes_call = sum(w.algorithmic_bytes for w in ws) / n_routes
    tot, slow = aggregate(dist, bytes_call * calls, sec)
    peak, peak_kind = measured_peak_gbs()
    gbs = tot / slow / 1e9
    return {
        "workload": f"grouped decode GEMV {name}: E={E} experts of M={M} K={K}, "
                    f"{workloads.GROUPED[name]['tokens']} tokens x top-"
                    f"{workloads.GROUPED[name]['top_k']} = {T} rows, {n_routes} routings rotated",
        "us_per_call": round(sec / calls * 1e6, 3), "calls": calls, "GB/s": round(gbs, 2),
        "frac": round(gbs / peak, 4), "peak_kind": f"{peak_kind} HBM copy bandwidth (burst)",
        "active_experts": [w.active_experts for w in ws],
        "bytes_per_call": int(bytes_call),
        "kernel": KERNEL_NAMES.get(pkg.nvfp4_gemv_plan(M, K, T).kernel, "?"),
        "weights_resident_mb": round((w0.A.nbytes + w0.sfa.nbytes) / 1e6, 1),
    }


def time_general(pkg, w, stream, steps, warmup, dist, n_copies):
    """The general path: the same workload with every input 1 byte past a 16-byte boundary, which
    the planner sends to the byte-load kernel (any alignment, any K % 16 == 0)."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    sets, keep = [], []
    for _ in range(n_copies):
        s = {}
        for k in ("A", "sfa", "b", "sfb"):
            x = np.ascontiguousarray(getattr(w, k)).ravel()
            raw = torch.empty(x.size + 32, dtype=torch.uint8, device=dev)
            v = raw[1:1 + x.size]
            v.copy_(torch.from_numpy(x))
            keep.append(raw)
            s[k] = v
        sets.append(s)
    outs = [torch.empty((w.L, w.M), dtype=torch.float16, device=dev) for _ in range(n_copies)]

    peak, _ = measured_peak_gbs()
    out = {"inputs": "A, sfa, b, sfb each 1 byte past a 16-byte boundary"}
    # the automatic plan in strict order and with early weights, then the byte-load kernel forced
    # on the same inputs
    for name, plan in (("automatic", None), ("automatic_early_weights", {"flags": FLAG_EARLY_WEIGHTS}),
                       ("byte_loads", {"kernel": 1})):
        def fn(i, plan=plan):
            s = sets[i % n_copies]
            pkg.nvfp4_gemv_batched_ex(s["A"], s["sfa"], w.g_a, s["b"], s["sfb"], w.g_b,
                                      outs[i % n_copies], w.M, w.K, w.L, stream=stream, plan=plan)
        sec, calls = _graph_time(fn, stream, steps, warmup, dist, dev)
        tot, slow = aggregate(dist, w.algorithmic_bytes * calls, sec)
        # the automatic plan for unaligned operands: the register-vector TMA kernel's unaligned
        # form when K % 256 == 0 and every CTA slot gets at least 8 rows, else the shift kernel
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        auto = (KERNEL_NAMES[4] + " (unaligned form)"
                if w.K % 256 == 0 and w.M * w.L // (2 * sms) >= 8 else KERNEL_NAMES[6])
        out[name] = {"kernel": KERNEL_NAMES[1] if plan and plan.get("kernel") == 1 else auto,
                     "us_per_call": round(sec / calls * 1e6, 3), "calls": calls,
                     "GB/s": round(tot / slow / 1e9, 2), "frac": round(tot / slow / 1e9 / peak, 4)}
    return out


def time_large(pkg, device, stream, steps, warmup, dist, M=7168, K=16384, L=80):
    """A many-batch call of the decode projection shape: 80 batches of 7168 x 16384 (5.29 GB per
    call, far larger than L2, so no rotation).  Batch q's A is one seeded block with every byte
    XORed with a per-batch key; every batch has its own vector.  The per-call start and drain
    are small against 0.7 ms of streaming, so this shows the kernel's streaming rate."""
    import torch

    blk = workloads.random_workload(M, K, 1, seed=31)
    vec = workloads.random_workload(1, K, L, seed=32)
    dA = torch.from_numpy(blk.A[0]).to(device)
    dS = torch.from_numpy(blk.sfa[0]).to(device)
    A = torch.empty((L, M, K // 2), dtype=torch.uint8, device=device)
    S = torch.empty((L, M, K // 16), dtype=torch.uint8, device=device)
    for q in range(L):
        torch.bitwise_xor(dA, (37 * q + 11) & 0xFF, out=A[q])
        S[q].copy_(dS)
    b = torch.from_numpy(vec.b).to(device)
    sfb = torch.from_numpy(vec.sfb).to(device)
    c = torch.empty((L, M), dtype=torch.float16, device=device)
    plan = {"flags": FLAG_EARLY_WEIGHTS}

    def fn(i):
        pkg.nvfp4_gemv_batched_ex(A, S, blk.g_a, b, sfb, vec.g_b, c, M, K, L, stream=stream,
                                  plan=plan)
    sec, calls = _graph_time(fn, stream, steps, warmup, dist, device)
    assert not torch.isnan(c).any().item()
    nbytes = workloads.algorithmic_bytes(M, K, L)
    gbs = nbytes * calls / sec / 1e9
    peak, _ = measured_peak_gbs()
    p = pkg.nvfp4_gemv_plan(M, K, L)
    del A, S
    torch.cuda.empty_cache()
    return {"workload": f"M={M} K={K} L={L} ({nbytes / 1e9:.2f} GB per call)",
            "kernel": KERNEL_NAMES.get(p.kernel), "ctas_per_batch": p.ctas_per_batch,
            "us_per_call": round(sec / calls * 1e6, 3), "calls": calls,
            "GB/s": round(gbs, 2), "frac": round(gbs / peak, 4)}


def time_small_n(pkg, device, stream, steps, warmup, dist, M=7168, K=16384, Ns=(2, 8, 16)):
    """N vectors sharing one weight matrix (a decode batch): the tensor-core kernel (automatic
    plan) against the register-vector CUDA-core kernel reading A once per vector.  Bytes: A and
    sfa once, the N vectors, the N output rows.  Weights rotate over copies larger than L2."""
    import torch

    w = workloads.random_workload(M, K, 1, seed=2, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    ncp = max(2, -(-3 * l2 // (M * K * 9 // 16)) + 1)
    As = [torch.from_numpy(w.A[0]).to(device) for _ in range(ncp)]
    Ss = [torch.from_numpy(w.sfa[0]).to(device) for _ in range(ncp)]
    peak, _ = measured_peak_gbs()
    out = {"workload": f"M={M} K={K}, N vectors sharing A (rotated over {ncp} copies)"}
    for N in Ns:
        v = workloads.random_workload(1, K, N, seed=3)
        b = torch.from_numpy(v.b).to(device)
        sb = torch.from_numpy(v.sfb).to(device)
        c = torch.empty((N, M), dtype=torch.float16, device=device)
        byt = M * K * 9 // 16 + N * K * 9 // 16 + 2 * M * N
        row = {}
        for name, plan in (("tensor_cores", {"flags": FLAG_EARLY_WEIGHTS}),
                           ("cuda_cores_rv", {"kernel": 4, "flags": FLAG_EARLY_WEIGHTS})):
            def fn(i, plan=plan):
                pkg.nvfp4_gemm_small_n(As[i % ncp], Ss[i % ncp], w.g_a, b, sb, w.g_b, c, M, K, N,
                                       stream=stream, plan=plan)
            sec, calls = _graph_time(fn, stream, steps, warmup, dist, device)
            gbs = byt * calls / sec / 1e9
            row[name] = {"us_per_call": round(sec / calls * 1e6, 3), "GB/s": round(gbs, 2),
                         "frac": round(gbs / peak, 4)}
        row["speedup"] = round(row["cuda_cores_rv"]["us_per_call"] /
                               row["tensor_cores"]["us_per_call"], 2)
        out[f"N={N}"] = row
    out["context_torch_scaled_mm"] = time_scaled_mm_context(device, stream, steps, warmup, dist,
                                                            As, Ss, M, K)
    return out


def time_scaled_mm_context(device, stream, steps, warmup, dist, As, Ss, M, K, N=16):
    """Context, not this library: the route the pages take for a small batch of tokens,
    torch._scaled_mm on NVFP4 operands (a cuBLASLt kernel), on the same rotated weight bytes and
    byte count.  Its vector side must be a multiple of 16, so N < 16 pads to 16 and costs the same.
    The block scales are one constant byte (1.0), so their tile layout does not matter: this times
    the call and compares no values."""
    import torch

    if not hasattr(torch, "float4_e2m1fn_x2"):
        return {"unavailable": "this torch has no float4_e2m1fn_x2 type"}
    rup = lambda x, m: (x + m - 1) // m * m
    ncp = len(As)
    a4 = [a.view(torch.float4_e2m1fn_x2) for a in As]
    sa = [torch.full((rup(M, 128) * rup(K // 16, 4),), 0x38, dtype=torch.uint8,
                     device=device).view(torch.float8_e4m3fn) for _ in range(ncp)]
    b = torch.from_numpy(workloads.random_workload(1, K, N, seed=3).b).to(device)
    b4 = b.view(torch.float4_e2m1fn_x2)
    sb = torch.full((rup(N, 128) * rup(K // 16, 4),), 0x38, dtype=torch.uint8,
                    device=device).view(torch.float8_e4m3fn)
    byt = M * K * 9 // 16 + N * K * 9 // 16 + 2 * M * N
    peak, _ = measured_peak_gbs()
    res = {"route": "torch._scaled_mm, NVFP4 operands (cuBLASLt), vector side padded to 16",
           "N": N, "values": "not compared (timing only)"}
    for name, od in (("fp16_out", torch.float16), ("bf16_out", torch.bfloat16)):
        try:
            def fn(i, od=od):
                torch._scaled_mm(a4[i % ncp], b4.t(), sa[i % ncp], sb, out_dtype=od)
            sec, calls = _graph_time(fn, stream, steps, warmup, dist, device)
        except Exception as ex:  # an older torch or a cuBLASLt without this path
            res[name] = {"unavailable": f"{type(ex).__name__}: {str(ex)[:120]}"}
            continue
        gbs = byt * calls / sec / 1e9
        res[name] = {"us_per_call": round(sec / calls * 1e6, 3), "GB/s": round(gbs, 2),
                     "frac": round(gbs / peak, 4)}
    return res


def time_tc_n1(pkg, w, sets, outs, stream, steps, warmup, dist, device):
    """The batched GEMV (N = 1 per batch) forced onto the tensor-core kernel, same inputs."""
    n = len(sets)
    plan = {"kernel": 5, "flags": FLAG_EARLY_WEIGHTS}

    def fn(i):
        s = sets[i % n]
        pkg.nvfp4_gemv_batched_ex(s["A"], s["sfa"], w.g_a, s["b"], s["sfb"], w.g_b, outs[i % n],
                                  w.M, w.K, w.L, stream=stream, plan=plan)
    sec, calls = _graph_time(fn, stream, steps, warmup, dist, device)
    gbs = w.algorithmic_bytes * calls / sec / 1e9
    peak, _ = measured_peak_gbs()
    return {"kernel": "gemv_tc_kernel", "us_per_call": round(sec / calls * 1e6, 3),
            "GB/s": round(gbs, 2), "frac": round(gbs / peak, 4),
            "plan": plan}


def run_ours(args):
    import torch

    import decode_nvfp4_gemv_gb300 as pkg

    world, rank, local = dist_env()
    dist = dist_init(world)
    if torch.cuda.device_count() <= local:
        raise SystemExit(f"rank {rank}: needs GPU {local}, this host has "
                         f"{torch.cuda.device_count()}")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pkg.load_library()
    w, name = headline_workload(args)
    bytes_call = w.algorithmic_bytes
    n_copies, l2 = _copies_for(bytes_call, device)
    sets = _device_inputs(w, n_copies, device)
    outs = [torch.empty((w.L, w.M), dtype=torch.float16, device=device) for _ in range(n_copies)]
    # Static weights: the same A and sfa are read by every call and written by none, so the calls
    # declare it (NVFP4_FLAG_EARLY_WEIGHTS) and each kernel starts streaming A while the previous
    # call drains.  The strict-order number (no flag) is reported beside it.
    plan = json.loads(args.plan) if args.plan else {"flags": FLAG_EARLY_WEIGHTS}
    stream = torch.cuda.Stream(device)
    timer = GraphTimer(_gemv_caller(pkg, w, sets, outs, plan, stream), args.steps, args.warmup,
                       stream)
    used_plan = plan_with_flags(pkg, w.M, w.K, w.L, plan)
    uuid = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"

    # the dominant kernel's launches on the launching stream: one per step
    sampler = ClockSampler(gpu_id)
    seconds = timer.time(dist, device, sampler)
    clocks = sampler.summary()

    total_bytes, slowest = aggregate(dist, bytes_call * args.steps, seconds)
    value = total_bytes / slowest / 1e9
    per_call_s = seconds / args.steps
    achieved = bytes_call / per_call_s / 1e9
    peak, peak_kind = measured_peak_gbs()
    traffic = recorded_traffic(name)

    # correctness spot check of the timed launches' last output (NaN would mean an unwritten c)
    assert not torch.isnan(outs[(args.steps - 1) % n_copies]).any().item()
    spread = timer.spread(device)
    chunk = timer.chunk
    del timer

    strict = None
    if not args.plan and not args.no_strict:
        steps_s = min(args.steps, 20000)
        t = GraphTimer(_gemv_caller(pkg, w, sets, outs, {"flags": 0}, stream), steps_s,
                       args.warmup, stream)
        sec_s = t.time(dist, device)
        del t
        tot_s, slow_s = aggregate(dist, bytes_call * steps_s, sec_s)
        strict = {"value": round(tot_s / slow_s / 1e9, 2), "unit": "GB/s",
                  "us_per_call": round(sec_s / steps_s * 1e6, 3), "steps": steps_s,
                  "frac": round(tot_s / slow_s / 1e9 / peak, 4),
                  "flags": "none (every read waits for the preceding call; the first ring fill "
                           "is prefetched into L2 before the wait, a hint that changes no value)"}
        t = GraphTimer(_gemv_caller(pkg, w, sets, outs, {"flags": FLAG_NO_L2_PREFETCH}, stream),
                       steps_s, args.warmup, stream)
        sec_n = t.time(dist, device)
        del t
        tot_n, slow_n = aggregate(dist, bytes_call * steps_s, sec_n)
        strict["without_l2_prefetch"] = {"us_per_call": round(sec_n / steps_s * 1e6, 3),
                                         "frac": round(tot_n / slow_n / 1e9 / peak, 4)}

    per_config = None
    if not args.plan and not args.no_per_config:
        per_config = time_per_config(pkg, device, stream, min(args.steps, 20000), args.warmup,
                                     dist)

    small_ml = None
    if not args.plan and not args.no_small_ml:
        small_ml = time_small_ml(pkg, device, stream, min(args.steps, 5000), args.warmup, dist)

    bf16 = None
    if not args.plan and not args.no_bf16:
        bf16 = time_bf16_vector(pkg, w, sets, outs, stream, min(args.steps, 20000), args.warmup,
                                dist)

    tc_n1 = None
    if not args.plan and not args.no_tc:
        tc_n1 = time_tc_n1(pkg, w, sets, outs, stream, min(args.steps, 20000), args.warmup, dist,
                           device)

    small = None
    if not args.plan and not args.no_tc:
        small = time_small_n(pkg, device, stream, min(args.steps, 5000), args.warmup, dist)

    general = None
    if not args.plan and not args.no_general:
        general = time_general(pkg, w, stream, min(args.steps, 2000), args.warmup, dist, n_copies)

    large = None
    if not args.plan and not args.no_large:
        large = time_large(pkg, device, stream, min(args.steps, 100), args.warmup, dist)

    grouped = None
    if not args.plan and not args.no_grouped:
        grouped = time_grouped(pkg, device, stream, min(args.steps, 20000), args.warmup, dist)

    e2e = None
    if not args.no_e2e:
        # host buffers are copied in before every call, so A is written by preceding work: no flag
        e2e = time_e2e(pkg, w, None, device, stream, min(args.steps, args.e2e_steps), dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(slowest / args.steps * 1e3, 6),
            "us_per_call": round(per_call_s * 1e6, 3),
            "us_per_call_spread": spread,
            "pct_of_peak": round(100.0 * achieved / peak, 2),
            "pct_of_nominal_hbm": round(100.0 * achieved / NOMINAL_HBM_GBS, 2),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "dtype_detail": "e2m1 / e4m3 inputs, exact f16x2 block sums, f32 scaling and "
                            "accumulation, f16 output",
            "data": "synthetic (seeded splitmix64; " + w.recipe + ")",
            "config": workload_config(w, name, world),
            "plan": used_plan,
            "launch": f"CUDA graphs of {chunk} calls after a spin-kernel pre-roll",
            "roofline": {
                "bound": "hbm",
                "kernel": KERNEL_NAMES.get(used_plan.get("kernel"), "?"),
                "achieved": round(achieved, 2),
                "peak": peak,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "peak_kind": f"{peak_kind} HBM copy bandwidth (burst)",
                "traffic": traffic,
            },
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        for key, val in (("strict_order", strict), ("per_config", per_config),
                         ("small_ml", small_ml), ("bf16_vector", bf16), ("grouped", grouped),
                         ("general_unaligned", general), ("large_batch", large),
                         ("tensor_cores_n1", tc_n1), ("small_n", small), ("e2e", e2e),
                         ("cpu_baseline", cpu)):
            if val is not None:
                line[key] = val
        print(json.dumps(line), flush=True)
    barrier(dist)


def time_e2e(pkg, w, plan, device, stream, steps, dist, copy_streams=1):
    """GB/s of algorithmic bytes when every step copies its inputs from pinned host memory, runs
    the GEMV through the public call and reads c back to pinned host memory.  The input copy of a
    step is split over `copy_streams` streams (the copy engines work in parallel) into one of two
    device buffers, so step i's copies overlap step i-1's GEMV and read-back; a buffer is reused
    only after the GEMV that read it has finished."""
    import torch

    names = ("A", "sfa", "b", "sfb")
    host = {k: torch.from_numpy(np.ascontiguousarray(getattr(w, k)).ravel()).pin_memory()
            for k in names}
    devb = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    c_dev = [torch.empty((w.L, w.M), dtype=torch.float16, device=device) for _ in range(2)]
    c_host = [torch.empty((w.L, w.M), dtype=torch.float16).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() for v in host.values())
    d2h = c_host[0].numel() * 2
    cps = [torch.cuda.Stream(device) for _ in range(copy_streams)]
    nA = host["A"].numel()
    cuts = [nA * j // copy_streams for j in range(copy_streams + 1)]
    done = [None, None]  # event after the GEMV that last read buffer 0 / 1

    def step(i, start=None):
        bi = i % 2
        evs = []
        for j, cs in enumerate(cps):
            if start is not None:
                cs.wait_event(start)
            if done[bi] is not None:
                cs.wait_event(done[bi])
            with torch.cuda.stream(cs):
                devb[bi]["A"][cuts[j]:cuts[j + 1]].copy_(host["A"][cuts[j]:cuts[j + 1]],
                                                         non_blocking=True)
                if j == copy_streams - 1:
                    for k in ("sfa", "b", "sfb"):
                        devb[bi][k].copy_(host[k], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            evs.append(ev)
        for ev in evs:
            stream.wait_event(ev)
        d = devb[bi]
        with torch.cuda.stream(stream):
            pkg.nvfp4_gemv_batched_ex(d["A"], d["sfa"], w.g_a, d["b"], d["sfb"], w.g_b,
                                      c_dev[bi], w.M, w.K, w.L, stream=stream, plan=plan)
            fin = torch.cuda.Event()
            fin.record(stream)
            done[bi] = fin
            c_host[bi].copy_(c_dev[bi], non_blocking=True)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(device)
    barrier(dist)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i, start=ev0 if i == 0 else None)
    ev1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist)
    seconds = ev0.elapsed_time(ev1) / 1e3
    total, slowest = aggregate(dist, w.algorithmic_bytes * steps, seconds)
    return {"value": round(total / slowest / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "us_per_step": round(seconds / steps * 1e6, 2),
            "copies": f"{copy_streams} streams, double-buffered inputs"}


# ---------------------------------------------------------------------------- the oracle on the CPU

def _row_bytes(w, n_rows):
    """Algorithmic bytes of n_rows outputs (their share of the vector bytes included)."""
    return w.algorithmic_bytes * n_rows / (w.M * w.L)


def _oracle_rows(w, start, n, threads):
    """The C oracle (fp64) on output rows start .. start+n-1 of the workload (wrapping around)."""
    from oracle import cref

    idx = (start + np.arange(n, dtype=np.int64)) % (w.M * w.L)
    ls, ms = np.divmod(idx, w.M)
    cref.gemv_rows(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L, ls, ms, threads=threads)


def _host_cpus():
    cpus = os.cpu_count() or 1
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return cpus, model


def _timed_rows(w, seconds, threads, chunk):
    """Rows computed by the C oracle in about `seconds` of wall time, and that time."""
    done = 0
    t0 = time.perf_counter()
    while True:
        _oracle_rows(w, done, chunk, threads)
        done += chunk
        el = time.perf_counter() - t0
        if el >= seconds:
            return done, el


def cpu_baseline(w, seconds: float):
    """The oracle as it stands (plain C, fp64, built with gcc -O2) timed on this host: one thread
    over consecutive output rows for a third of `seconds`, then an OpenMP parallel for over output
    rows on every host thread for the rest; both wrap around the workload, a bounded sample of
    about `seconds` of CPU time."""
    from oracle import cref

    total = w.M * w.L
    chunk1 = max(1, (1 << 21) // w.K)
    rows1, el1 = _timed_rows(w, seconds / 3, 1, chunk1)
    single = {"value": round(_row_bytes(w, rows1) / el1 / 1e9, 4), "cores": 1,
              "sample": f"{rows1} output rows ({rows1 / total:.2f} x the workload) in {el1:.1f} s"}
    threads = cref.max_threads()
    cpus, model = _host_cpus()
    rows, el = _timed_rows(w, seconds * 2 / 3, threads, max(threads * 8, (1 << 24) // w.K))
    return {"value": round(_row_bytes(w, rows) / el / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{rows} output rows ({rows / total:.2f} x the workload, wrapping) in "
                      f"{el:.1f} s, plain C fp64 oracle, OpenMP parallel for over rows on "
                      f"{threads} threads",
            "host_cpus": cpus, "host_cpu_model": model, "single_thread": single}


def run_reference(args):
    """The oracle as it stands (plain C, fp64, OpenMP over output rows on every host thread), each
    step a bounded sample of consecutive output rows of the workload, sized so that the whole
    run fits --reference-seconds.  Under several ranks rank 0 alone runs it."""
    from oracle import cref

    world, rank, _ = dist_env()
    if rank != 0:
        return
    w, name = headline_workload(args)
    total = w.M * w.L
    threads = cref.max_threads()
    per_step_budget = args.reference_seconds / max(1, args.steps + args.warmup)
    probe = max(threads, 64)
    t0 = time.perf_counter()
    _oracle_rows(w, 0, probe, threads)
    t_row = max((time.perf_counter() - t0) / probe, 1e-7)
    rows = int(max(threads, min(4 * total, per_step_budget / t_row)))
    for i in range(args.warmup):
        _oracle_rows(w, i * rows, rows, threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_rows(w, (args.warmup + i) * rows, rows, threads)
    elapsed = time.perf_counter() - t0
    value = _row_bytes(w, rows) * args.steps / elapsed / 1e9
    cpus, model = _host_cpus()
    sample = (f"{rows} consecutive output rows per step (wrapping) of the M={w.M} K={w.K} L={w.L} "
              f"workload, plain C fp64 oracle, OpenMP parallel for over rows on {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, name, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample, "host_cpus": cpus,
                             "host_cpu_model": model},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--config", default="c2", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--shape", default="",
                    help="time any M x K x L instead of --config (e.g. 8192x65536x1)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--plan", default="", help="JSON plan fields forced on every call")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-strict", action="store_true",
                    help="skip the second timing without the early-weights flag")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the timings of all five decode workloads")
    ap.add_argument("--no-small-ml", action="store_true",
                    help="skip the few-rows / long-K (split-K) timings")
    ap.add_argument("--no-bf16", action="store_true",
                    help="skip the bf16-vector (activation quantization) timing")
    ap.add_argument("--no-grouped", action="store_true",
                    help="skip the grouped (mixture-of-experts) timing")
    ap.add_argument("--no-general", action="store_true",
                    help="skip the unaligned-input (byte-load kernel) timing")
    ap.add_argument("--no-large", action="store_true",
                    help="skip the 80-batch (5.29 GB per call) timing")
    ap.add_argument("--no-tc", action="store_true",
                    help="skip the tensor-core timings (N = 1 and small N)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.shape:
        try:
            parse_shape(args.shape)
        except ValueError as e:
            ap.error(str(e))
    world_env = os.environ.get("WORLD_SIZE")
    if world_env is not None and int(world_env) != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world_env}: launch one rank per GPU")
    if world_env is None and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
