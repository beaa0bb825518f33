#!/usr/bin/env python
"""Benchmark of the chunked tensor-parallel MLP on GB300.

One step = one pass of the whole hot path over one batch of synthetic input: for the default
workload (Llama-3 8B-shaped SwiGLU MLP, M = 8 x 4096 tokens, h = 4096, ffn = 14336, t = 8 shards,
p = 2 row chunks) the forward (first linear + SwiGLU, second linear into per-shard fp32 partials,
shard-sum) and the backward (output-gradient GEMM with SwiGLU backward, weight gradients
accumulated into fp32, input-gradient partials and their shard-sum).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line on rank 0.  ``value`` is GEMM TFLOP/s of the whole job (all ranks) with
inputs resident in HBM; ``e2e`` is the same metric with the per-step host->device copy of the
activations (X, gY) from pinned memory and the device->host read of the step's outputs (Y, gX)
inside the timed region.  ``--impl reference`` times the CPU oracle on a bounded sample.
With N > 1 every rank runs an independent replica (the emulated shards live on one GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from comm_overlap_gb300 import synth  # noqa: E402

METRIC = "TFLOP/s of chunked TP-shard MLP fwd+bwd on 1 GB300; % of dense BF16 peak"
DEFAULT_WORKLOAD = "llama3_8b_swiglu_fwdbwd"
ACT_NAMES = {0: "none", 1: "relu", 2: "gelu", 3: "swiglu", 4: "bilinear"}

# The sources each kernel kind is built from: a kind's ncu traffic (below) is reported only while
# the code of these files (comments excluded) hashes as it did when the traffic was captured.
KIND_SOURCES = {"gemm": ("gemm.cuh", "ptx.cuh", "actfn.cuh"), "elementwise": ("elementwise.cu", "actfn.cuh"),
                "attention": ("attention.cu", "ptx.cuh")}


def source_group(kernel: str) -> str:
    if kernel.startswith("gemm_"):
        return "gemm"
    return "attention" if kernel == "attention" else "elementwise"


# DRAM traffic per launch from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum), keyed by
# workload and kernel kind, with the hash of the kind's sources at capture time.
# Captured one kernel and one launch at a time on a small case of the workload (M = 8192 tokens in
# one row chunk, m = 8192 per launch) and scaled x 2 to the m = 16384 launch of the full workload:
# only kinds whose reduction length does not grow with the tokens are listed, since their traffic
# grows in proportion to the rows a launch processes.  The weight-gradient GEMMs reduce over the
# tokens, so theirs does not scale that way and is left out (reported null).  The second linear of
# the default schedule runs once as the fp32-partial kernel (1.448 GB at m = 8192) and, for the
# call's last chunk, once as the fused shard-sum kernel (1.111 GB): its entry is the mean per launch.
_SHA_GEMM = "18acfe21c2ea6673"
_SHA_ELEM = "6a7ca743efb34cd0"
NCU_TRAFFIC = {
    ("llama3_8b_swiglu_fwdbwd", "gemm_fwd1"): {"bytes_per_launch": 2 * 1.454e9, "src_sha": _SHA_GEMM},
    ("llama3_8b_swiglu_fwdbwd", "gemm_fwd2"): {"bytes_per_launch": 2 * 1.2795e9, "src_sha": _SHA_GEMM},
    ("llama3_8b_swiglu_fwdbwd", "shard_sum"): {"bytes_per_launch": 2 * 1.092e9, "src_sha": _SHA_ELEM},
    ("llama3_8b_swiglu_fwdbwd", "gemm_dgrad_h"): {"bytes_per_launch": 2 * 2.111e9, "src_sha": _SHA_GEMM},
    ("llama3_8b_swiglu_fwdbwd", "gemm_dgrad_x"): {"bytes_per_launch": 2 * 2.315e9, "src_sha": _SHA_GEMM},
}


def _code_only(text: str) -> str:
    """Source text without comments and blank lines, so that comment edits keep the hash."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_sha(group: str = "gemm") -> str:
    """SHA-256 (16 hex digits) of the code, comments excluded, of the sources of one kernel group
    (KIND_SOURCES)."""
    h = hashlib.sha256()
    for f in KIND_SOURCES[group]:
        with open(os.path.join(ROOT, "comm_overlap_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
               "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "source": "measured"}
        # the median SM clock under which the sustained peak was measured, for per-clock comparisons
        mhz = (d.get("clocks_under_load") or {}).get("sm_mhz_median")
        if mhz:
            out["sustained_sm_mhz"] = float(mhz)
        return out
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 50 ms while the timed region runs.  Each row carries nvidia-smi's own
    timestamp; `stop(t0, t1)` keeps the rows whose time falls inside the host-side window of the
    timed loop (the GPU is busy for all of it: the host only enqueues, then waits at the barrier),
    so an idle lead-in or tail does not enter the median."""

    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # let nvidia-smi initialise before the timed region starts
        deadline = time.time() + 3.0
        while time.time() < deadline and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
            time.sleep(0.05)

    def stop_raw(self):
        """Stops sampling; the rows taken (csv text, None when nvidia-smi could not be started)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.path) as fh:
            text = fh.read()
        os.unlink(self.path)
        return text

    def stop(self, t0=None, t1=None):
        text = self.stop_raw()
        if text is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        return summarize_clocks(text, t0, t1)


def _smi_time(stamp: str):
    """Seconds since the epoch of an nvidia-smi timestamp ("2026/12/02 11:25:03.123", local time)."""
    import datetime
    try:
        return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


def _num(v: str):
    try:
        return float(v)
    except ValueError:
        return None


def summarize_clocks(text: str, t0=None, t1=None) -> dict:
    """Median SM clock, maximum clock, throttle reasons and peak power of the nvidia-smi rows in
    `text` (ClockSampler.FIELDS, csv, no header) whose timestamps fall in [t0, t1] (all rows when no
    window is given).  `samples` counts the rows used; `in_window` says whether the window held any
    (if not, every row is used and the record says so)."""
    rows = []
    for line in text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) == len(ClockSampler.FIELDS):
            rows.append(dict(zip(ClockSampler.FIELDS, parts)))
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    use, in_window = rows, None
    if t0 is not None and t1 is not None:
        win = [r for r in rows if (_smi_time(r["timestamp"]) or -1.0) >= t0 and (_smi_time(r["timestamp"]) or 1e30) <= t1]
        in_window = bool(win)
        if win:
            use = win
    sm = sorted(v for v in (_num(r["clocks.sm"]) for r in use) if v is not None)
    power = [v for v in (_num(r["power.draw"]) for r in use) if v is not None]
    reasons = sorted({name for r in use for name in ClockSampler.REASONS
                      if r["clocks_event_reasons." + name].lower() == "active"})
    out = {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": _num(use[0]["clocks.max.sm"]),
           "reasons": reasons, "samples": len(use), "power_w_max": max(power) if power else None}
    if in_window is not None:
        out["in_window"] = in_window
    return out


def physical_gpu(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


# ------------------------------------------------------------------------------ multi-rank timing

def max_over_ranks(values, world: int, device: str):
    """Element-wise maximum of per-rank timings (the slowest rank sets the job's time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tflops(flops_per_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs `steps` steps of `flops_per_step` in `ms` (max over ranks)."""
    return world * steps * flops_per_step / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------------------ workload

def kernel_work(s: synth.MlpShape):
    """Algorithmic flops (GEMMs) or bytes (HBM kernels) per launch of each kernel kind."""
    m, n = s.M // s.p, s.h // s.q
    a_rows = s.a_rows
    return {
        "gemm_fwd1": ("tensor", 2.0 * m * s.h * a_rows),
        "gemm_fwd2": ("tensor", 2.0 * m * s.F * n),
        "shard_sum": ("hbm", s.t * m * n * 4.0 + m * n * 2.0 + (m * n * 2.0 if s.layernorm else 0.0)),
        "layernorm": ("hbm", 2.0 * m * s.h * 2.0),
        "gemm_dgrad_h": ("tensor", 2.0 * m * s.h * s.F),
        "gemm_wgrad_b": ("tensor", 2.0 * m * s.h * s.F),
        "gemm_dgrad_x": ("tensor", 2.0 * m * (2 * s.F if s.gated else s.F) * n),
        "gemm_wgrad_a": ("tensor", 2.0 * m * (2 * s.F if s.gated else s.F) * s.h),
        "layernorm_bwd": ("hbm", 4.0 * m * s.h * 2.0 + m * 4.0),
        "gemm_qkv": ("tensor", 2.0 * m * s.h * 3 * s.h),
        # q.k and p.v over the visible (causal) key positions: 4 d per pair, seq (seq + 1) / 2 pairs
        # per sequence and head
        "attention": ("tensor", 4.0 * s.h * m * (s.seq + 1) / 2.0),
        "gemm_oproj": ("tensor", 2.0 * m * s.h * n),
    }


def config_json(s: synth.MlpShape, sched: str, n_gpus: int, reduce_ctas: int = 0):
    c = {"workload": s.name, "M": s.M, "batch": s.batch, "seq": s.seq, "h": s.h, "ffn": s.F,
         "act": ACT_NAMES[s.act], "t": s.t, "p": s.p, "q": s.q, "layers": s.layers, "heads": s.heads,
         "layernorm": s.layernorm, "pass": "fwd+bwd" if s.backward else "fwd", "sched": sched,
         "seed": 0, "l2": "inputs larger than L2 (129 MB); no flush needed",
         "parallelism": "replicas" if n_gpus > 1 else "single GPU, t shards emulated in HBM"}
    if reduce_ctas:
        c["reduce_ctas"] = reduce_ctas
    return c


# ------------------------------------------------------------------------------ CPU baseline

def oracle_sample(s: synth.MlpShape, inp: dict, scale: float = 1.0, min_units: int = 1):
    """Times the CPU oracle on a bounded sample of the workload; returns (flops, seconds, what).
    Every sampled quantity (token rows, gradient rows, ffn features) counts at least `min_units`
    items, so that with min_units = the oracle's thread count no thread sits idle."""
    import oracle
    X, A, B = inp["X"], inp["A"], inp["B"]
    fwd_row = 2.0 * s.h * s.a_rows + 2.0 * s.F * s.h

    def count(k):
        return max(min_units, int(round(k * scale)))

    n_fwd = max(2, count(24))
    rows = synth.sample_indices(s.M, n_fwd, 1)
    flops = 0.0
    t0 = time.perf_counter()
    if s.attention:
        # causality: the first positions of one sequence do not depend on the rest of it
        upto = max(2, count(12))
        oracle.block_fwd(X, inp["Wqkv"], inp["Wo"], A, B, s.t, s.heads, s.seq, s.act, 1e-5, seqs=[0], upto=upto)
        attn_row = 2.0 * s.h * 4 * s.h + 4.0 * s.h * (upto + 1) / 2.0
        flops += upto * (fwd_row + attn_row) * s.layers
        what = f"the first {upto} positions of one sequence through all {s.layers} blocks"
    elif s.layernorm:
        oracle.stack_fwd(X, A, B, s.t, s.act, 1e-5, rows=rows)
        flops += len(rows) * fwd_row * s.layers
        what = f"{len(rows)} token rows through all {s.layers} layers"
    else:
        oracle.mlp_fwd(X, A[0], B[0], s.t, s.act, rows=rows)
        flops += len(rows) * fwd_row
        what = f"forward of {len(rows)} token rows"
    if s.backward and s.layernorm:
        n_b = count(4)
        rows_b = synth.sample_indices(s.M, n_b, 2)
        oracle.stack_bwd(X, A, B, inp["gY"], s.t, s.act, 1e-5, rows=rows_b)
        # forward again (the row backward recomputes it) plus dH and dX per layer
        flops += len(rows_b) * s.layers * (fwd_row + 2.0 * s.h * s.F + 2.0 * s.h * s.a_rows)
        what += f"; input gradient of {len(rows_b)} rows through all {s.layers} layers"
    elif s.backward:
        n_dx = count(8)
        n_ft = count(24)
        rows_b = synth.sample_indices(s.M, n_dx, 2)
        feats = synth.sample_indices(s.F, n_ft, 3)
        oracle.mlp_bwd(X, A[0], B[0], inp["gY"], s.t, s.act, rows=rows_b, want_dw=False)
        oracle.mlp_bwd(X, A[0], B[0], inp["gY"], s.t, s.act, feats=feats, want_dx=False)
        flops += len(rows_b) * (2.0 * s.h * s.F + 2.0 * s.h * s.a_rows)  # dH and dX of those rows
        flops += len(feats) * (2.0 * s.M * s.h * (3 if s.gated else 2))  # dA rows and dB column over all M
        what += f"; input gradient of {len(rows_b)} rows; weight gradients of {len(feats)} ffn features over all M"
    dt = time.perf_counter() - t0
    return flops, dt, what


def reduction_roofline(kern: dict, work: dict, peaks: dict, workload: str, alone_ms=None):
    """The shard-sum (the AllReduce stand-in) against the HBM roofline: algorithmic bytes per launch
    over its event duration, live (concurrent with the GEMMs of the next chunk, sharing HBM with
    them) and, when measured, alone on the same sizes.  Null when the schedule fuses the reduction
    into the GEMM."""
    k = kern.get("shard_sum")
    if not k or not k["launches"]:
        return None
    nbytes = work["shard_sum"][1]
    avg_ms = k["total_ms"] / k["launches"]
    gbs = nbytes / (avg_ms * 1e-3) / 1e9
    out = {"bound": "hbm", "kernel": "shard_sum", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": avg_ms,
           "concurrent_with_gemms": True, "traffic": traffic_per_launch(workload, "shard_sum")}
    if alone_ms:
        alone = nbytes / (alone_ms * 1e-3) / 1e9
        out["alone"] = {"achieved": alone, "frac": alone / peaks["hbm_gbs"], "avg_launch_ms": alone_ms}
    return out


def shard_sum_alone(s: synth.MlpShape, stream, reps: int = 10):
    """Average duration (ms) of the shard-sum alone, on the workload's partial size (t x m x n fp32
    in, m x n bf16 out, plus the residual for layer stacks), timed with CUDA events."""
    import torch

    from comm_overlap_gb300 import domino as dm
    m, n = s.M // s.p, s.h // s.q
    P = torch.randn(s.t, m, n, device="cuda")
    Y = torch.empty((m, s.h), dtype=torch.bfloat16, device="cuda")
    res = torch.zeros((m, s.h), dtype=torch.bfloat16, device="cuda") if s.layernorm else None
    for _ in range(3):
        dm.domino_shard_sum(P, s.t, m, n, res, s.h, Y, s.h, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        dm.domino_shard_sum(P, s.t, m, n, res, s.h, Y, s.h, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del P, Y, res
    torch.cuda.empty_cache()
    return ms


def traffic_per_launch(workload: str, kernel: str, sha: str | None = None):
    """ncu DRAM bytes per launch of a kernel on a workload, if captured on the current code of the
    kernel's sources (`sha`: that code's hash, computed when not given)."""
    t = NCU_TRAFFIC.get((workload, kernel))
    if t is None:
        return None
    if sha is None:
        sha = kernel_source_sha(source_group(kernel))
    return t["bytes_per_launch"] if t.get("src_sha") == sha else None


def fp8_inputs(s: synth.MlpShape) -> dict:
    """E4M3 codes of the workload's draws with power-of-two per-tensor scales: X ~ N(0, 1) at 2^-6,
    the weights ~ N(0, 0.02) at 2^-11, and the first-linear output at 2^-6 (GeLU) or 2^-5 (SwiGLU),
    which keep |value / scale| inside the E4M3 range 448."""
    sx, sw = 2.0 ** -6, 2.0 ** -11
    sh = 2.0 ** -5 if s.gated else 2.0 ** -6
    return {"X": synth.e4m3_codes((s.M, s.h), s.x_std, sx, 0, synth.TID_X),
            "A": synth.e4m3_codes((s.a_rows, s.h), s.w_std, sw, 0, synth.TID_A),
            "B": synth.e4m3_codes((s.t, s.h, s.Fi), s.w_std, sw, 0, synth.TID_B),
            "scales": (sx, sw, sw, sh)}


def oracle_sample_fp8(s: synth.MlpShape, inp: dict, scale: float = 1.0, min_units: int = 1):
    import oracle
    rows = synth.sample_indices(s.M, max(2, min_units, int(round(24 * scale))), 1)
    t0 = time.perf_counter()
    oracle.mlp_fwd_fp8(inp["X"], inp["A"], inp["B"], s.t, s.act, inp["scales"], rows=rows)
    dt = time.perf_counter() - t0
    flops = len(rows) * (2.0 * s.h * s.a_rows + 2.0 * s.F * s.h)
    return flops, dt, f"FP8 forward of {len(rows)} token rows"


# ------------------------------------------------------------------------------ exposed reduction

def reduction_alone_ms(trace, reduce_kind: int) -> tuple[float, float]:
    """From a launch timeline [(kind, start_ms, end_ms), ...]: the summed time of the `reduce_kind`
    launches, and the part of it during which no launch of another kind ran (the reduction left
    exposed on the timeline)."""
    others = sorted((a, b) for k, a, b in trace if k != reduce_kind and b > a)
    merged = []
    for a, b in others:
        if merged and a <= merged[-1][1]:
            merged[-1][1] = max(merged[-1][1], b)
        else:
            merged.append([a, b])
    total = alone = 0.0
    for k, a, b in trace:
        if k != reduce_kind or b <= a:
            continue
        total += b - a
        covered = sum(max(0.0, min(b, y) - max(a, x)) for x, y in merged if x < b and y > a)
        alone += (b - a) - covered
    return total, alone


def exposure_summary(windows: list, steps: int) -> dict:
    """Exposed reduction from alternating timed windows: `windows` holds (arm, ms for `steps` steps,
    median SM MHz) with arm "normal" or "noreduce".  The exposed time is the step-time difference of
    the medians; `frac` divides it by the normal step time.  `frac_equal_clock` compares SM cycles
    (time x median MHz) instead, removing the part of the difference that comes from the clock the
    power cap allowed each arm."""
    import statistics

    def med(arm, i):
        v = [w[i] for w in windows if w[0] == arm and w[i] is not None]
        return statistics.median(v) if v else None

    t_n, t_0 = med("normal", 1) / steps, med("noreduce", 1) / steps
    f_n, f_0 = med("normal", 2), med("noreduce", 2)
    out = {"frac": (t_n - t_0) / t_n, "ms": t_n - t_0, "ms_per_step_normal": t_n, "ms_per_step_noreduce": t_0,
           "sm_mhz_normal": f_n, "sm_mhz_noreduce": f_0, "steps_per_window": steps,
           "windows": [{"arm": a, "ms_per_step": ms / steps, "sm_mhz": f} for a, ms, f in windows]}
    if f_n and f_0:
        out["frac_equal_clock"] = (t_n * f_n - t_0 * f_0) / (t_n * f_n)
    return out


# ------------------------------------------------------------------------------ our arm

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from comm_overlap_gb300 import build as cuda_build
    from comm_overlap_gb300 import domino as dm

    if rank == 0 or not os.path.exists(cuda_build.LIB):
        cuda_build.build()
    if world > 1:
        torch.distributed.barrier()
    s = args.shape
    sched = {"serial": dm.SCHED_SERIAL, "intra": dm.SCHED_INTRA, "inter": dm.SCHED_INTER,
             "fused": dm.SCHED_FUSED}[args.sched]
    fp8 = args.fp8
    if fp8 and (s.backward or s.layernorm or s.attention):
        raise SystemExit("--fp8 runs the single-MLP forward workloads (add --pass fwd for the fwd+bwd one)")
    inp = synth.make_inputs(s, seed=0) if not fp8 else fp8_inputs(s)

    def dev(a):
        if a.dtype == np.uint8:
            return torch.from_numpy(np.ascontiguousarray(a)).cuda()
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    X, A, B = dev(inp["X"]), dev(inp["A"]), dev(inp["B"])
    gY = dev(inp["gY"]) if s.backward else None
    h = dm.domino_create()
    cfg = dm.make_cfg(s.M, s.h, s.F, s.t, s.p, s.q, s.act, sched=sched, layers=s.layers, ln_eps=1e-5,
                      heads=s.heads, seq=s.seq if s.attention else 0, reduce_ctas=args.reduce_ctas)
    Wqkv = dev(inp["Wqkv"]) if s.attention else None
    Wo = dev(inp["Wo"]) if s.attention else None
    if fp8:
        wsb = dm.domino_workspace_size(cfg, dm.PASS_FWD_FP8)
    elif s.attention:
        wsb = dm.domino_workspace_size(cfg, dm.PASS_BLOCK)
    elif s.layernorm:
        wsb = max(dm.domino_workspace_size(cfg, dm.PASS_STACK),
                  dm.domino_workspace_size(cfg, dm.PASS_STACK_BWD) if s.backward else 0)
    else:
        wsb = max(dm.domino_workspace_size(cfg, dm.PASS_FWD),
                  dm.domino_workspace_size(cfg, dm.PASS_BWD) if s.backward else 0)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    Y = torch.empty((s.M, s.h), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((s.M, s.a_rows), dtype=torch.bfloat16, device="cuda") if s.backward and not s.layernorm else None
    save = (torch.empty(dm.domino_stack_save_size(cfg), dtype=torch.uint8, device="cuda")
            if s.backward and s.layernorm else None)
    gX = torch.empty_like(Y) if s.backward else None
    gA = torch.zeros((s.layers * s.a_rows, s.h), dtype=torch.float32, device="cuda") if s.backward else None
    gB = torch.zeros((s.layers * s.t, s.h, s.Fi), dtype=torch.float32, device="cuda") if s.backward else None
    stream = torch.cuda.current_stream()

    def step_on(st, Xin, gYin, Yout=None, gXout=None):
        Yout = Y if Yout is None else Yout
        gXout = gX if gXout is None else gXout
        if fp8:
            dm.domino_mlp_fwd_fp8(h, cfg, Xin, A, B, inp["scales"], Yout, ws, wsb, st)
            return
        if s.attention:
            dm.domino_block_fwd(h, cfg, Xin, Wqkv, Wo, A, B, Yout, ws, wsb, st)
            return
        if s.layernorm:
            if s.backward:
                dm.domino_stack_fwd_train(h, cfg, Xin, A, B, Yout, save, ws, None, wsb, st)
                dm.domino_stack_bwd(h, cfg, A, B, save, gYin, gXout, gA, gB, ws, None, wsb, st)
            else:
                dm.domino_stack_fwd(h, cfg, Xin, A, B, Yout, ws, wsb, st)
            return
        dm.domino_mlp_fwd(h, cfg, Xin, A, B, Yout, S, ws, wsb, st)
        if s.backward:
            dm.domino_mlp_bwd(h, cfg, Xin, A, B, S, gYin, gXout, gA, gB, ws, wsb, st)

    def step(Xin, gYin):
        step_on(stream, Xin, gYin)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step(X, gY)
    barrier()

    # ---- device-resident timing (the `value`), per-kernel events on their own streams
    clocks = ClockSampler(physical_gpu(local_rank))
    clocks.start()
    dm.domino_timing_reset(h)
    dm.domino_timing_enable(h, True)
    n_launch0 = dm.domino_launch_count(h)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_loop0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step(X, gY)
    e1.record(stream)
    barrier()
    t_loop1 = time.time()
    clk = clocks.stop(t_loop0, t_loop1)
    dm.domino_timing_enable(h, False)
    launches = dm.domino_launch_count(h) - n_launch0
    ms = e0.elapsed_time(e1)
    ms_eager = ms
    if args.graph:
        # one step captured as a CUDA graph (the eager steps above did the one-time set-up),
        # replayed `steps` times; the per-kernel timings come from the eager pass above
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step_on(side, X, gY)
        for _ in range(args.warmup):
            graph.replay()
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        barrier()
        ms = e0.elapsed_time(e1)
    kern = {}
    for k, name in enumerate(dm.KERNEL_NAMES):
        n, tot = dm.domino_timing_read(h, k)
        if n:
            kern[name] = {"launches": n, "total_ms": tot}
    # the timed steps' launch timeline: how much of the shard-sum time ran with no other kernel
    timeline = None
    if "shard_sum" in kern:
        tot, alone = reduction_alone_ms(dm.domino_timing_trace(h), dm.K_SHARD_SUM)
        timeline = {"shard_sum_ms_per_step": tot / args.steps, "alone_ms_per_step": alone / args.steps,
                    "hidden_frac": 1.0 - alone / tot if tot > 0 else None,
                    "source": "CUDA events around every launch on its own stream (domino_timing_trace), "
                              "timed steps of the value"}

    # ---- exposed reduction: the same schedule with every shard-sum replaced by a kernel that does
    # no reduction (domino_debug_skip_reduce), in windows of >= exposure_s seconds alternating with
    # the normal path, clocks sampled in each window
    exposed = None
    if args.exposure and args.sched == "fused":
        exposed = {"frac": None, "why": "FUSED reduces inside the GEMMs; the no-reduce variant applies to the "
                                        "stream schedules"}
    elif args.exposure:
        per_step = max_over_ranks([ms_eager], world, "cuda")[0] / args.steps   # the same count on every rank
        n_win = max(3, int(-(-args.exposure_s * 1e3 // per_step)))
        sampler = ClockSampler(physical_gpu(local_rank))
        sampler.start()
        spans = []
        for arm in ("normal", "noreduce") * args.exposure_pairs:
            dm.domino_debug_skip_reduce(h, arm == "noreduce")
            for _ in range(3):
                step(X, gY)
            barrier()
            w0 = time.time()
            e0.record(stream)
            for _ in range(n_win):
                step(X, gY)
            e1.record(stream)
            barrier()
            spans.append((arm, e0.elapsed_time(e1), w0, time.time()))
        dm.domino_debug_skip_reduce(h, False)
        raw = sampler.stop_raw()
        wins = [(a, max_over_ranks([w_ms], world, "cuda")[0],
                 summarize_clocks(raw, w0, w1).get("sm_mhz") if raw else None) for a, w_ms, w0, w1 in spans]
        exposed = exposure_summary(wins, n_win)
        exposed["method"] = ("T_step - T_step(no-reduce): the same schedule with every shard-sum launch replaced "
                             "by a same-grid kernel that does no reduction (residual copy in layer stacks) and the "
                             "call's last chunk on the plain partial GEMM; medians of alternating windows")
    if exposed is not None or timeline is not None:
        exposed = dict(exposed or {})
        exposed["timeline"] = timeline
    st, site = dm.domino_device_status(h)
    if st != 0:
        raise RuntimeError(f"device error word set during the benchmark: {site:#x}")

    # ---- end to end through the C ABI: every step copies its inputs (X, gY) from pinned host
    # memory and reads its outputs (Y, gX) back.  As a training loop would, the next step's inputs
    # are prefetched on one copy stream while the current step computes, and each step's outputs
    # are read back on another while the next step computes (double-buffered device buffers).
    hX = (torch.from_numpy(inp["X"]) if fp8 else torch.from_numpy(inp["X"].view(np.int16)).view(torch.bfloat16))
    hX = hX.pin_memory()
    hgY = torch.from_numpy(inp["gY"].view(np.int16)).view(torch.bfloat16).pin_memory() if s.backward else None
    hY = torch.empty((s.M, s.h), dtype=torch.bfloat16).pin_memory()
    hgX = torch.empty((s.M, s.h), dtype=torch.bfloat16).pin_memory() if s.backward else None
    Xs = [torch.empty_like(X) for _ in range(2)]
    gYs = [torch.empty_like(gY) for _ in range(2)] if s.backward else [None, None]
    Ys = [Y, torch.empty_like(Y)]
    gXs = [gX, torch.empty_like(gX)] if s.backward else [None, None]
    h2d = hX.numel() * hX.element_size() + (hgY.numel() * 2 if s.backward else 0)
    d2h = hY.numel() * 2 + (hgX.numel() * 2 if s.backward else 0)
    cs_in, cs_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]

    def prefetch(b):
        with torch.cuda.stream(cs_in):
            Xs[b].copy_(hX, non_blocking=True)
            if s.backward:
                gYs[b].copy_(hgY, non_blocking=True)
            ev_in[b].record(cs_in)

    def e2e_steps(n):
        cs_in.wait_stream(stream)
        cs_out.wait_stream(stream)
        prefetch(0)
        for k in range(n):
            b = k % 2
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_read[b])  # step k-2's outputs have been read back
            step_on(stream, Xs[b], gYs[b], Ys[b], gXs[b])
            ev_done[b].record(stream)
            if k + 1 < n:
                if k >= 1:
                    cs_in.wait_event(ev_done[1 - b])  # step k-1 no longer reads buffer 1-b
                prefetch(1 - b)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(ev_done[b])
                hY.copy_(Ys[b], non_blocking=True)
                if s.backward:
                    hgX.copy_(gXs[b], non_blocking=True)
                ev_read[b].record(cs_out)
        stream.wait_stream(cs_in)
        stream.wait_stream(cs_out)

    e2e_steps(max(2, args.warmup // 2))
    clocks_e2e = ClockSampler(physical_gpu(local_rank))
    clocks_e2e.start()
    barrier()
    t_e2e0 = time.time()
    e0.record(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    barrier()
    t_e2e1 = time.time()
    clk_e2e = clocks_e2e.stop(t_e2e0, t_e2e1)
    ms_e2e = e0.elapsed_time(e1)
    dm.domino_destroy(h)
    ss_alone = shard_sum_alone(s, stream) if "shard_sum" in kern and not fp8 else None

    ms, ms_e2e = max_over_ranks([ms, ms_e2e], world, "cuda")
    if rank != 0:
        return None

    flops = s.gemm_flops()
    value = job_tflops(flops, args.steps, world, ms)
    e2e = job_tflops(flops, args.steps, world, ms_e2e)
    peaks = load_peaks()
    work = kernel_work(s)
    dom = max(kern, key=lambda k: kern[k]["total_ms"])
    bound, per_launch = work[dom]
    avg_ms = kern[dom]["total_ms"] / kern[dom]["launches"]
    sha = {g: kernel_source_sha(g) for g in KIND_SOURCES}
    traffic_val = traffic_per_launch(s.name, dom)
    # FP8 contractions: the measured bf16 peak times the nominal dense ratio 4.5 / 2.25 = 2.  The
    # sustained (power-capped) peak applies when the run hit the power cap; a run that held its
    # clocks (short steps) is held to the burst figure.
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    peak_key = "bf16_tflops_sustained" if capped else "bf16_tflops"
    peak_scale = 2.0 if fp8 else 1.0
    peak_kind = ("e4m3 = 2 x " if fp8 else "") + ("bf16 sustained" if capped else "bf16 burst")
    if bound == "tensor":
        achieved = per_launch / (avg_ms * 1e-3) / 1e12
        peak = peaks[peak_key] * peak_scale
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_val,
                "peak_kind": f"{peak_kind} ({peaks['source']})", "algorithmic_flops_per_launch": per_launch,
                "avg_launch_ms": avg_ms}
    else:
        achieved = per_launch / (avg_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic_val, "peak_kind": f"hbm copy ({peaks['source']})",
                "algorithmic_bytes_per_launch": per_launch, "avg_launch_ms": avg_ms}
    # the same fraction per SM cycle: a kernel that ran at another clock than the one the sustained
    # peak was measured at is compared at equal clocks (TFLOP/s per MHz)
    if bound == "tensor" and clk.get("sm_mhz") and peaks.get("sustained_sm_mhz"):
        per_mhz_peak = peaks["bf16_tflops_sustained"] * peak_scale / peaks["sustained_sm_mhz"]
        roof["per_clock"] = {"frac": achieved / clk["sm_mhz"] / per_mhz_peak, "sm_mhz": clk["sm_mhz"],
                             "peak_sm_mhz": peaks["sustained_sm_mhz"],
                             "note": "achieved / run clock over sustained peak / its clock"}
    total_k = sum(v["total_ms"] for v in kern.values())
    for name, v in kern.items():
        b, w = work[name]
        v["share"] = v["total_ms"] / total_k
        v["avg_ms"] = v["total_ms"] / v["launches"]
        if b == "tensor":
            v["tflops"] = w / (v["avg_ms"] * 1e-3) / 1e12
        else:
            v["gbs"] = w / (v["avg_ms"] * 1e-3) / 1e9
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16", "data": "synthetic",
           "config": config_json(s, args.sched, world, args.reduce_ctas),
           "pct_of_peak": {"of_sustained": value / world / (peaks["bf16_tflops_sustained"] * peak_scale),
                           "of_burst": value / world / (peaks["bf16_tflops"] * peak_scale),
                           "peaks": peaks["source"] + (" x 2 for e4m3" if fp8 else "")},
           "roofline": roof,
           "reduction": reduction_roofline(kern, work, peaks, s.name, ss_alone),
           "e2e": {"value": e2e, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "sm_mhz": clk_e2e.get("sm_mhz"), "clock_reasons": clk_e2e.get("reasons")},
           "gpu_launches": launches, "clocks": clk, "kernels": kern, "kernel_src_sha": sha}
    if fp8:
        out["config"]["operands"] = "e4m3 with per-tensor scales (sx, sa, sb, sh) = " + str(inp["scales"])
    if args.graph:
        out["config"]["graph"] = True
        out["eager_value"] = world * args.steps * flops / (ms_eager * 1e-3) / 1e12
    if world == 1 and not args.no_cpu_baseline:
        flops_s, dt, what = (oracle_sample_fp8 if fp8 else oracle_sample)(s, inp, scale=5.0)
        import oracle
        out["cpu_baseline"] = {"value": flops_s / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                               "kind": "oracle", "sample": what, "seconds": dt}
    out["exposed"] = exposed
    return out


# ------------------------------------------------------------------------------ reference arm

def run_reference(args, rank):
    if rank != 0:
        return None
    s = args.shape
    inp = synth.make_inputs(s, seed=0)
    import oracle
    oracle.lib()
    # each step: one item per oracle thread of every sampled quantity (rows, ffn features), so the
    # host's cores all work; about a second per step on 16 cores for the fwd+bwd workload
    threads = oracle.num_threads()
    for _ in range(args.warmup):
        oracle_sample(s, inp, scale=0.1, min_units=threads)
    total_f, total_t, what = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, dt, what = oracle_sample(s, inp, scale=0.1, min_units=threads)
        total_f += f
        total_t += dt
    value = total_f / total_t / 1e12
    cores = oracle.num_threads()
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_json(s, args.sched, 1, getattr(args, "reduce_ctas", 0)),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: " + what},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.SHAPES))
    ap.add_argument("--sched", default="intra", choices=["serial", "intra", "inter", "fused"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pass", dest="pass_", default=None, choices=["fwd", "fwd+bwd"],
                    help="override the workload's pass (profiling aid)")
    ap.add_argument("--p", type=int, default=None, help="override the row-chunk count")
    ap.add_argument("--q", type=int, default=None, help="override the column-chunk count")
    ap.add_argument("--M", type=int, default=None, help="override the token count (profiling aid)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true", help="time replays of one step captured as a CUDA graph")
    ap.add_argument("--fp8", action="store_true", help="E4M3 operands (domino_mlp_fwd_fp8), forward MLP workloads")
    ap.add_argument("--no-exposure", dest="exposure", action="store_false",
                    help="skip the exposed-reduction leg (normal vs no-reduce windows)")
    ap.add_argument("--exposure-s", dest="exposure_s", type=float, default=1.1,
                    help="seconds per timed window of the exposed-reduction leg")
    ap.add_argument("--exposure-pairs", dest="exposure_pairs", type=int, default=2,
                    help="normal / no-reduce window pairs of the exposed-reduction leg")
    ap.add_argument("--reduce-ctas", dest="reduce_ctas", type=int, default=0,
                    help="CTAs per shard-sum launch (cfg.reduce_ctas; 0 = the library default)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    import dataclasses
    s = synth.SHAPES[args.workload]
    over = {}
    if args.pass_ is not None:
        over["backward"] = args.pass_ == "fwd+bwd"
    if args.p is not None:
        over["p"] = args.p
    if args.q is not None:
        over["q"] = args.q
    if args.M is not None:
        over["M"] = args.M
    args.shape = dataclasses.replace(s, **over) if over else s
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        import torch
        torch.cuda.set_device(local_rank)
        if world > 1:
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        try:
            out = run_ours(args, rank, world, local_rank)
        finally:
            if world > 1:
                torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
