"""Benchmark of the sliding-window attention hot path on GB300: one step = forward + backward
(Delta preprocess, dK/dV, dQ) of one long-context sliding-window layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (default): B=1, Hq=32, Hkv=16, N=32768, D=128, window 1024, bf16 Q/K/V ~ N(0,1),
dO ~ N(0, 1e-2), seeded synthetic data.  Metric: window-effective TFLOP/s of forward + backward,
counting only visible (query, key) pairs: forward 4*D, backward 10*D flops per pair and head.

Printed as one JSON line (rank 0).  `value` is device-timed with inputs resident in HBM; `e2e` is
the same metric with the host->device copy of the step's inputs and the device->host copy of its
outputs inside the timed region; `roofline` reports the dominant kernel against the measured peak;
`cpu_baseline` times the fp64 oracle on a bounded sample of the same workload on the host cores.
With --gpus N > 1 (launched under torchrun) every rank runs its own independent layer (weak
scaling, no data-path collective); the barrier and max-over-ranks timing use torch.distributed.
"""
from __future__ import annotations

import argparse
import dataclasses
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
import torch  # noqa: E402

import swa_inputs as si  # noqa: E402

METRIC = "SWA fwd+bwd window-effective TFLOP/s & peak GB at N=32768, W=1024 (1×GB300)"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------------------------------------
# Flop and byte accounting (window-effective: visible pairs only)
# ------------------------------------------------------------------------------------------------

def visible_pairs(N: int, W: int) -> int:
    """(query, key) pairs with 0 <= i - j < W in one head of length N."""
    W = min(W, N)
    return N * W - W * (W - 1) // 2


def window_pairs(Lq: int, Lk: int, W: int, causal: bool) -> int:
    """Visible (query, key) pairs in one head when query i sits at key position i + Lk - Lq and
    sees keys j with 0 <= pos - j < W (causal) or |pos - j| < W (two-sided)."""
    pos = np.arange(Lq, dtype=np.int64) + (Lk - Lq)
    lo = np.maximum(pos - (W - 1), 0)
    hi = pos if causal else np.minimum(pos + (W - 1), Lk - 1)
    return int(np.sum(hi - lo + 1))


def step_flops(case: si.Case) -> dict:
    pairs = visible_pairs(case.N, case.W) * case.B * case.Hq
    return {
        "fwd": 4 * case.D * pairs,
        "bwd": 10 * case.D * pairs,
        # algorithmic share of each backward kernel: dK/dV does the S, dP, dV and dK contractions
        # of the backward's five, dQ adds the fifth (its own S and dP are recomputation)
        "dkdv": 8 * case.D * pairs,
        "dq": 2 * case.D * pairs,
        "pairs": pairs,
    }


def delta_bytes(case: si.Case) -> int:
    rows = case.B * case.Hq * case.N
    return rows * case.D * 2 * 2 + rows * 4


def aggregate_tflops(world: int, flops_per_step_per_rank: int, steps: int, ms_max: float) -> float:
    """Whole-job window-effective TFLOP/s: every rank ran `steps` steps of the same workload
    (weak scaling); the job took the slowest rank's time."""
    return world * flops_per_step_per_rank * steps / (ms_max * 1e-3) / 1e12


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ------------------------------------------------------------------------------------------------

_CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
_CLOCK_PERIOD_MS = 10  # the timed region of the default run is ~40 ms: sample densely


def _smi_time(stamp: str):
    """Seconds since the epoch of an nvidia-smi timestamp ('YYYY/MM/DD HH:MM:SS.mmm', local)."""
    import datetime

    try:
        return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


class ClockSampler:
    """nvidia-smi polling in the background while the timed region runs.  `mark(start, end)` gives
    the wall-clock bounds of the timed region; the summary keeps the samples inside it (or, when
    none landed inside, the ones at most one period from it) and says how many there were."""

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={_CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(_CLOCK_PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self, start: float, end: float):
        self.window = (start, end)

    def __exit__(self, *exc):
        time.sleep(2 * _CLOCK_PERIOD_MS / 1000)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def _parsed(self):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        rows = []
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {n for n, val in zip(names, parts[6:10]) if val.lower().startswith("active")}
            rows.append((_smi_time(parts[0]), sm, mx, reasons))
        return rows

    def summary(self) -> dict:
        rows = self._parsed()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sel, where = rows, "whole sampler run"
        if self.window is not None:
            t0, t1 = self.window
            inside = [r for r in rows if r[0] is not None and t0 <= r[0] <= t1]
            slack = _CLOCK_PERIOD_MS / 1000
            near = [r for r in rows if r[0] is not None and t0 - slack <= r[0] <= t1 + slack]
            if inside:
                sel, where = inside, "inside the timed region"
            elif near:
                sel, where = near, f"within {_CLOCK_PERIOD_MS} ms of the timed region"
        reasons = sorted(set().union(*(r[3] for r in sel)))
        return {"sm_mhz": statistics.median(r[1] for r in sel),
                "sm_max_mhz": max(r[2] for r in sel), "reasons": reasons, "samples": len(sel),
                "sm_mhz_min": min(r[1] for r in sel), "period_ms": _CLOCK_PERIOD_MS,
                "selection": where, "samples_total": len(rows)}


# ------------------------------------------------------------------------------------------------
# Distributed plumbing (barrier and max-over-ranks only)
# ------------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, device):
    if world <= 1:
        return None
    import torch.distributed as dist

    backend = "nccl" if device.type == "cuda" else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device):
    if dist is not None:
        if device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# The CPU oracle on a bounded sample
# ------------------------------------------------------------------------------------------------

def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_sample(case: si.Case, rows_per_sample: int, samples: int, seed: int = 0) -> dict:
    """Time the fp64 oracle (forward + backward) on `samples` blocks of `rows_per_sample` query rows
    of head (0, 0) of the workload, mid-sequence; returns window-effective TFLOP/s of that work."""
    from oracle import swa_oracle as orc

    import numpy as np

    N, D, W = case.N, case.D, case.W
    one_head = si.Case(B=1, Hq=1, Hkv=1, N=N, D=D, W=W, do_std=case.do_std, seed=seed)
    inp = si.make_inputs(one_head)
    qh, kh, vh, doh = (inp[k_][0, 0].double().numpy() for k_ in ("q", "k", "v", "do"))

    flops = 0
    t0 = time.perf_counter()
    for s in range(samples):
        r0 = min(N - rows_per_sample, N // 2 + s * rows_per_sample) if N > rows_per_sample else 0
        rows = np.arange(r0, min(N, r0 + rows_per_sample))
        orc.rows_backward(qh, kh, vh, doh, rows, W, case.softmax_scale)
        vis = int(np.sum(np.minimum(rows + 1, W)))
        flops += 14 * D * vis
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "seconds": dt, "flops": flops,
            "rows": rows_per_sample * samples}


def cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo; Arm hosts name no model there)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_info() -> dict:
    return {"cpu_model": cpu_model(), "cpu_count": os.cpu_count(), "blas_threads": _blas_threads(),
            "note": "BLAS matmuls use blas_threads threads; NumPy's elementwise ops use one"}


def _group_rows_seconds(case: si.Case, rows_per_head: int) -> dict:
    """The oracle's forward + backward of kv group 0 (kv head 0 of batch 0 and its G query heads):
    the whole group when rows_per_head >= N, else `rows_per_head` consecutive mid-sequence rows of
    each of the group's heads.  The dense oracle's cost is the same for every row (it scores every
    key), so the whole group's time is the sample's time x N / rows."""
    from oracle import swa_oracle as orc

    G = case.Hq // case.Hkv
    one_group = si.Case(B=1, Hq=G, Hkv=1, N=case.N, D=case.D, W=case.W, do_std=case.do_std,
                        seed=case.seed)
    inp = si.make_inputs(one_group)
    R = min(rows_per_head, case.N)
    r0 = (case.N - R) // 2
    rows = np.arange(r0, r0 + R)
    heads = [(inp["q"][0, g].double().numpy(), inp["do"][0, g].double().numpy()) for g in range(G)]
    k0, v0 = inp["k"][0, 0].double().numpy(), inp["v"][0, 0].double().numpy()
    t0 = time.perf_counter()
    for qh, doh in heads:
        if R == case.N:
            orc.head_backward(qh, k0, v0, doh, case.W, case.softmax_scale)
        else:
            orc.rows_backward(qh, k0, v0, doh, rows, case.W, case.softmax_scale)
    dt = time.perf_counter() - t0
    group_s = dt * case.N / R
    return {"measured_s": dt,
            "measured": ("whole kv group" if R == case.N else
                         f"{R} mid-sequence rows of each of the kv group's {G} query heads"),
            "group_s" if R == case.N else "group_s_extrapolated": group_s,
            "all_heads_s_extrapolated": group_s * case.B * case.Hkv}


def cpu_baselines(gpu_ms: dict, rows_per_head: int = 2048) -> dict:
    """The fp64 oracle beside each workload's GPU time: the full oracle for the tiny case and the
    edge sweep, one kv group (measured, or a row sample of it) for the long layers, the full-causal
    GQA layer and the mixed step, with the all-heads (all-layers) time extrapolated and labelled."""
    from oracle import swa_oracle as orc

    out = {"host": host_info()}
    c = si.tiny_case()
    inp = si.make_inputs(c)
    t0 = time.perf_counter()
    orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], c.W, c.softmax_scale)
    out["tiny"] = {"oracle_s": time.perf_counter() - t0, "measured": "full oracle fwd + bwd",
                   "gpu_ms": gpu_ms.get("tiny")}
    t0 = time.perf_counter()
    for c in si.edge_cases():
        inp = si.make_inputs(c)
        orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], c.W, c.softmax_scale)
    out["edge_sweep"] = {"oracle_s": time.perf_counter() - t0, "cases": len(si.edge_cases()),
                         "measured": "full oracle fwd + bwd of every case",
                         "gpu_ms": gpu_ms.get("edge_sweep")}
    for N in (8192, 16384, 32768):
        case = si.long_swa_case(N)
        r = _group_rows_seconds(case, N if N == 8192 else rows_per_head)
        r["gpu_ms"] = gpu_ms.get(f"long_swa_{N}")
        out[f"long_swa_{N}"] = r
    r = _group_rows_seconds(si.gqa_causal_case(), 8192)
    r["gpu_ms"] = gpu_ms.get("gqa_causal_8k")
    out["gqa_causal_8k"] = r
    layers = si.mixed_layer_cases()
    per = [_group_rows_seconds(layers[i], rows_per_head) for i in (0, 5)]  # a sliding, a full layer
    n_full = sum(1 for c in layers if c.W >= c.N)
    tot = per[0]["all_heads_s_extrapolated"] * (len(layers) - n_full) + \
        per[1]["all_heads_s_extrapolated"] * n_full
    out["mixed_12_layers"] = {
        "measured_s": per[0]["measured_s"] + per[1]["measured_s"],
        "measured": f"{rows_per_head} mid-sequence rows of each query head of kv group 0, in one "
                    "sliding and one full layer",
        "layer_group_s_extrapolated": [per[0]["group_s_extrapolated"],
                                       per[1]["group_s_extrapolated"]],
        "all_layers_all_heads_s_extrapolated": tot,
        "gpu_ms": gpu_ms.get("mixed_12_layers"),
    }
    return out


# ------------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------------

def headline_config(case: si.Case, world: int) -> dict:
    """The `config` of both arms' JSON lines: the long sliding-window layer at N = 32,768."""
    fl = step_flops(case)
    return {
        "workload": f"long-context sliding-window layer: B={case.B} Hq={case.Hq} Hkv={case.Hkv} "
                    f"N={case.N} D={case.D} W={case.W}, fwd + bwd (Delta, dK/dV, dQ)",
        "B": case.B, "Hq": case.Hq, "Hkv": case.Hkv, "N": case.N, "D": case.D, "W": case.W,
        "global_batch": case.B * world,
        "seq_len": case.N,
        "parallelism": f"independent layer per rank x{world}" if world > 1 else "single GPU",
        "l2": f"no flush: each step reads Q/dO ({case.B * case.Hq * case.N * case.D * 2 / 1e6:.0f} "
              f"MB each) and K/V ({case.B * case.Hkv * case.N * case.D * 2 / 1e6:.0f} MB each), "
              "all larger than the 129 MB L2" if case.N >= 32768 else
              "no flush (a profiling size: the per-tensor footprint may fit in the 129 MB L2)",
        "flops_per_step": {"fwd": fl["fwd"], "bwd": fl["bwd"]},
    }


def run_ours(args, world, rank, local):
    import sliding_window_flash_gb300 as swa

    swa.load()  # fails loudly when libswa.so is missing: there is no fallback
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = dist_init(world, device)
    case = dataclasses.replace(si.long_swa_case(args.seq_len), D=args.head_dim)
    case = si.Case(**{**case.__dict__, "seed": rank})
    fl = step_flops(case)
    peaks = load_peaks()

    inp = si.make_inputs(case, device=str(device))
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    o = torch.empty_like(q)
    lse = torch.empty(case.B, case.Hq, case.N, dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty(case.B, case.Hq, case.N, dtype=torch.float32, device=device)
    ws_fused = torch.empty(swa.swa_attn_bwd_fused_workspace_bytes(case.B, case.Hq, case.N, case.D),
                           dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    # kernels of one step, in launch order (the backward's three phases after the forward)
    names = {"fused": ("fwd", "delta", "fused", "dq_convert"),
             "split": ("fwd", "delta", "dkdv", "dq")}

    def one_step(path, evs=None):
        if evs is not None:
            evs[0].record(stream)
        swa.swa_attn_fwd(q, k, v, case.W, case.softmax_scale, out=o, lse=lse)
        marks = None
        if evs is not None:
            marks = lambda i: evs[i + 1].record(stream)
        if path == "fused":
            swa.swa_attn_bwd_phases(q, k, v, o, do, lse, case.W, case.softmax_scale, dq=dq, dk=dk,
                                    dv=dv, between=marks, fused=True, workspace=ws_fused)
        else:
            swa.swa_attn_bwd_phases(q, k, v, o, do, lse, case.W, case.softmax_scale, dq=dq, dk=dk,
                                    dv=dv, delta=delta, between=marks)

    def timed_steps(path, steps, clk=None):
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier(dist, device)
        torch.cuda.synchronize(device)
        wall0 = time.time()
        start.record(stream)
        for s_ in range(steps):
            one_step(path, events[s_])
        end.record(stream)
        torch.cuda.synchronize(device)
        if clk is not None:
            clk.mark(wall0, time.time())
        barrier(dist, device)
        swa.swa_check_device(device)
        per = {n: [] for n in names[path]}
        for evs in events:
            for i, n in enumerate(names[path]):
                per[n].append(evs[i].elapsed_time(evs[i + 1]))
        return start.elapsed_time(end), {n_: sum(v_) / len(v_) for n_, v_ in per.items()}

    path = args.bwd
    for _ in range(args.warmup):
        one_step(path)
    torch.cuda.synchronize(device)
    swa.swa_check_device(device)
    with ClockSampler(local) as clk:
        total_ms, avg = timed_steps(path, args.steps, clk)
    total_ms = max_over_ranks(dist, total_ms, device)
    ms_step = total_ms / args.steps
    step_total = fl["fwd"] + fl["bwd"]
    value = aggregate_tflops(world, step_total, args.steps, total_ms)
    bwd_ms = sum(avg[n] for n in names[path][1:])

    kern_tflops = {"fwd": fl["fwd"] / (avg["fwd"] * 1e-3) / 1e12,
                   "bwd": fl["bwd"] / (bwd_ms * 1e-3) / 1e12}
    if path == "fused":
        kern_tflops["fused"] = fl["bwd"] / (avg["fused"] * 1e-3) / 1e12
    else:
        kern_tflops["dkdv"] = fl["dkdv"] / (avg["dkdv"] * 1e-3) / 1e12
        kern_tflops["dq"] = fl["dq"] / (avg["dq"] * 1e-3) / 1e12
    dominant = max((n for n in names[path] if n in kern_tflops), key=lambda k_: avg[k_])
    clocks = clk.summary()
    # The kernels run inside a short region (tens of ms) at the maximum SM clock, which is how the
    # burst peak was measured; the sustained peak comes from seconds of back-to-back GEMMs under
    # the power cap at a lower clock.  So the fraction is taken against the burst figure.
    peak_tf = peaks["bf16_tflops"]
    # the committed counters are of the headline layer's kernels
    traffic = _profiled_traffic(dominant) if (case.N, case.D) == (32768, 128) else None
    q_bytes = case.B * case.Hq * case.N * case.D * 2
    k_bytes = case.B * case.Hkv * case.N * case.D * 2
    row_bytes = case.B * case.Hq * case.N * 4
    acc_bytes = case.B * case.Hq * ((case.N + 127) // 128) * 128 * case.D * 4
    algorithmic_bytes = {  # each kernel's compulsory DRAM traffic per launch
        "fwd": 2 * q_bytes + 2 * k_bytes + row_bytes,
        "dkdv": 2 * q_bytes + 4 * k_bytes + 2 * row_bytes,
        "dq": 3 * q_bytes + 2 * k_bytes + 2 * row_bytes,
        # as dK/dV, plus reading and writing back the fp32 dQ accumulator (which the L2 cannot hold)
        "fused": 2 * q_bytes + 4 * k_bytes + 2 * row_bytes + 2 * acc_bytes,
    }
    # An even number of query heads per kv head runs the forward and dQ on CTA pairs at D = 128
    # and 256; D = 256 has kernels of its own (dK and dV two of them, always on CTA pairs).
    pair = case.D in (128, 256) and (case.Hq // case.Hkv) % 2 == 0
    if case.D == 256:
        kernel_names = {"fwd": "swa_fwd256_pair_kernel" if pair else "swa_fwd256_kernel",
                        "dkdv": "swa_dv256_pair_kernel + swa_dk256_pair_kernel",
                        "dq": "swa_dq256_pair_kernel" if pair else "swa_dq256_kernel",
                        "fused": "swa_fused_bwd_kernel<256>"}
    else:
        kernel_names = {"fwd": f"swa_fwd_pair_kernel<{case.D}>" if pair else f"swa_fwd_kernel<{case.D}>",
                        "dkdv": f"swa_dkdv_kernel<{case.D}>",
                        "dq": f"swa_dq_pair_kernel<{case.D}>" if pair else f"swa_dq_kernel<{case.D}>",
                        "fused": f"swa_fused_bwd_kernel<{case.D}>"}
    dom_flops = fl["bwd"] if dominant == "fused" else fl[dominant]
    roofline = {
        "kernel": kernel_names[dominant],
        "bound": "tensor",
        "achieved": kern_tflops[dominant],
        "peak": peak_tf,
        "unit": "TFLOP/s",
        "frac": kern_tflops[dominant] / peak_tf,
        "traffic": traffic,
        "algorithmic_bytes": algorithmic_bytes[dominant],
        "algorithmic_flops": dom_flops,
        "launch_ms": avg[dominant],
        "peak_source": f"{peaks['source']} bf16 burst (the kernel runs inside a "
                       f"{total_ms:.0f} ms region at {clocks.get('sm_mhz')} MHz)",
        "frac_of_sustained": kern_tflops[dominant] / peaks["bf16_tflops_sustained"]
        if peaks.get("bf16_tflops_sustained") else None,
    }
    if clocks.get("sm_mhz"):
        # clock-normalised duration: a kernel slowed only by a lower clock keeps this figure
        roofline["launch_kcycles"] = avg[dominant] * clocks["sm_mhz"]
    # The timed region is short (~40 ms at the default 20 steps), so only a few clock samples land
    # in it; the same step then runs untimed for ~0.5 s under the sampler, to show the clock that
    # this load holds (reported beside the timed region's samples, not instead of them).
    clocks_soak = None
    if not args.no_soak:
        with ClockSampler(local) as soak:
            soak_steps = max(1, int(500.0 / max(ms_step, 1e-3)))
            torch.cuda.synchronize(device)
            w0 = time.time()
            for _ in range(soak_steps):
                one_step(path)
            torch.cuda.synchronize(device)
            soak.mark(w0, time.time())
        clocks_soak = soak.summary()
        clocks_soak["steps"] = soak_steps
    # the other backward path, timed the same way right after (reported, not the headline; the
    # fused backward has no D = 256 form)
    other = "split" if path == "fused" else "fused"
    bwd_other = None
    if case.D != 256:
        for _ in range(3):
            one_step(other)
        o_ms, o_avg = timed_steps(other, args.steps)
        o_bwd = sum(o_avg[n] for n in names[other][1:])
        bwd_other = {"path": other, "ms_per_step": o_ms / args.steps, "kernels_ms": o_avg,
                     "bwd_ms": o_bwd, "bwd_tflops": fl["bwd"] / (o_bwd * 1e-3) / 1e12,
                     "fwd_bwd_tflops": step_total / (o_ms / args.steps * 1e-3) / 1e12}
        if other == "split":
            bwd_other["kernels_tflops"] = {"dkdv": fl["dkdv"] / (o_avg["dkdv"] * 1e-3) / 1e12,
                                           "dq": fl["dq"] / (o_avg["dq"] * 1e-3) / 1e12}
    # the fused path's preprocess also zeroes the fp32 dQ accumulator (acc_bytes written)
    delta_gbs = (delta_bytes(case) + (acc_bytes if path == "fused" else 0)) / \
        (avg["delta"] * 1e-3) / 1e9

    result = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(case, world),
        "gpu_launches": 4 * args.steps,
        "bwd_path": path,
        "kernels_ms": avg,
        "kernels_tflops": kern_tflops,
        "fwd_tflops": kern_tflops["fwd"],
        "bwd_tflops": kern_tflops["bwd"],
        "delta_gbs": delta_gbs,
        "roofline": roofline,
        "clocks": clocks,
        "clocks_soak": clocks_soak,
        "bwd_other_path": bwd_other,
    }

    if rank == 0 and not args.no_memory:
        result["memory"] = measure_memory(swa, device)
        result["peak_gb"] = result["memory"]["peak_gb_total"][-1]
        result["memory_fused_bwd"] = measure_memory(swa, device, fused=True)
        # the same layer with 256-wide heads, the shape of the pages' backward-memory figure
        result["memory_d256"] = measure_memory(swa, device, D=256)
    if not args.no_e2e:
        result["e2e"] = measure_e2e(swa, case, device, dist, args, world)
    if rank == 0 and not args.no_extra:
        result["other_workloads"] = measure_other_workloads(swa, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gpu_ms = measure_small_configs(swa, device)
        if "memory" in result:
            for N, ms in zip(result["memory"]["N"], result["memory"]["fwd_bwd_ms"]):
                gpu_ms[f"long_swa_{N}"] = ms
        gpu_ms.setdefault("long_swa_32768", ms_step)
        ow = result.get("other_workloads", {})
        if "gqa_causal_8k" in ow:
            gpu_ms["gqa_causal_8k"] = ow["gqa_causal_8k"]["fwd_ms"] + ow["gqa_causal_8k"]["bwd_ms"]
        if "mixed_12_layers" in ow:
            gpu_ms["mixed_12_layers"] = ow["mixed_12_layers"]["step_ms"]
        per = cpu_baselines(gpu_ms, rows_per_head=args.cpu_rows)
        result["cpu_baseline_per_config"] = per
        smp = per["long_swa_32768"]
        G = case.Hq // case.Hkv
        pairs = args.cpu_rows * case.W * G  # mid-sequence rows each see the whole window
        result["cpu_baseline"] = {
            "value": 14 * case.D * pairs / smp["measured_s"] / 1e12, "unit": UNIT,
            "cores": per["host"]["blas_threads"], "kind": "oracle",
            "sample": f"fp64 NumPy oracle fwd + bwd of {args.cpu_rows} mid-sequence query rows of "
                      f"each of the {G} query heads of one kv group of the N=32768 W=1024 layer, "
                      f"{smp['measured_s']:.1f} s (window-effective flops of those rows); "
                      "BLAS matmuls threaded, elementwise ops single-threaded",
            "seconds": smp["measured_s"],
            "cpu_model": per["host"]["cpu_model"], "cpu_count": per["host"]["cpu_count"],
        }
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu capture, or None when the kernel's sources
    have changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            ent = json.load(f).get(kernel)
        if not ent:
            return None
        h = hashlib.sha256()
        for name in ent["sources"]:
            with open(os.path.join(ROOT, "sliding_window_flash_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != ent["source_sha256"]:
            return None
        return ent["bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def measure_small_configs(swa, device) -> dict:
    """GPU fwd + bwd time of the tiny case (mean of 20 calls) and of the whole edge sweep (every
    case once, after one untimed pass), on preallocated buffers."""
    stream = torch.cuda.current_stream(device)
    out = {}

    def run(cases, reps):
        calls = []
        for c in cases:
            inp = si.make_inputs(c, device=str(device))
            calls.append(_layer_calls(swa, inp, c.W, c.softmax_scale))
        for f, b in calls:
            f()
            b()
        torch.cuda.synchronize(device)
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            for f, b in calls:
                f()
                b()
        e.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(e) / reps

    out["tiny"] = run([si.tiny_case()], 20)
    out["edge_sweep"] = run(si.edge_cases(), 1)
    swa.swa_check_device(device)
    return out


def measure_memory(swa, device, D: int = 128, fused: bool = False) -> dict:
    """Peak device memory of one layer's fwd + bwd versus N (inputs Q, K, V, dO excluded), for the
    long sliding-window layer with head dim D, and the fwd + bwd time at each N, on the split
    (default) or the fused backward."""
    out = {"D": D, "bwd_path": "fused" if fused else "split", "N": [], "peak_gb_total": [],
           "peak_gb_above_inputs": []}
    for N in (8192, 16384, 32768):
        case = dataclasses.replace(si.long_swa_case(N), D=D)
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
        before = torch.cuda.memory_allocated(device)  # what the process holds besides this layer
        inp = si.make_inputs(case, device=str(device))
        torch.cuda.synchronize(device)
        torch.cuda.reset_peak_memory_stats(device)
        base = torch.cuda.memory_allocated(device)
        o, lse = swa.swa_attn_fwd(inp["q"], inp["k"], inp["v"], case.W, case.softmax_scale)
        dq, dk, dv = swa.swa_attn_bwd(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, case.W,
                                      case.softmax_scale, fused=fused)
        torch.cuda.synchronize(device)
        peak = torch.cuda.max_memory_allocated(device)
        # time of one fwd + bwd at this length (after the memory-tracked one; 5 repetitions)
        nws = (swa.swa_attn_bwd_fused_workspace_bytes if fused else
               swa.swa_attn_bwd_workspace_bytes)(case.B, case.Hq, N, D)
        ws = torch.empty(nws, dtype=torch.uint8, device=device)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(5):
            swa.swa_attn_fwd(inp["q"], inp["k"], inp["v"], case.W, case.softmax_scale, out=o,
                             lse=lse)
            swa.swa_attn_bwd(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, case.W,
                             case.softmax_scale, dq=dq, dk=dk, dv=dv, workspace=ws, fused=fused)
        ev[1].record()
        torch.cuda.synchronize(device)
        ms = ev[0].elapsed_time(ev[1]) / 5
        fl = step_flops(case)
        out.setdefault("fwd_bwd_ms", []).append(ms)
        out.setdefault("fwd_bwd_tflops", []).append((fl["fwd"] + fl["bwd"]) / (ms * 1e-3) / 1e12)
        out["N"].append(N)
        out["peak_gb_total"].append((peak - before) / 1e9)  # the layer's inputs + fwd + bwd
        out["peak_gb_above_inputs"].append((peak - base) / 1e9)
        del inp, o, lse, dq, dk, dv, ws
    a = out["peak_gb_above_inputs"]
    out["ratio_per_doubling"] = [a[i + 1] / a[i] for i in range(len(a) - 1)]
    torch.cuda.empty_cache()
    return out


def measure_e2e(swa, case, device, dist, args, world) -> dict:
    """Same metric through the public host-buffer call (swa_attn_fwd_bwd_host): each step copies
    Q, K, V, dO from pinned host memory and O, LSE, dQ, dK, dV back to pinned host memory, the
    library pipelining those copies with the kernels over chunks of (batch, kv head) groups."""
    host = {k_: v_.cpu().pin_memory() for k_, v_ in si.make_inputs(case, device=str(device)).items()}
    outs = (torch.empty_like(host["q"]).pin_memory(),
            torch.empty((case.B, case.Hq, case.N), dtype=torch.float32).pin_memory(),
            torch.empty_like(host["q"]).pin_memory(), torch.empty_like(host["k"]).pin_memory(),
            torch.empty_like(host["v"]).pin_memory())
    U = swa.default_units_per_chunk(case.B, case.Hkv)
    ws = torch.empty(swa.swa_attn_host_workspace_bytes(case.B, case.Hq, case.Hkv, case.N, case.D, U),
                     dtype=torch.uint8, device=device)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)

    def step():
        swa.swa_attn_fwd_bwd_host(host["q"], host["k"], host["v"], host["do"], case.W,
                                  case.softmax_scale, outs=outs, units_per_chunk=U, workspace=ws,
                                  device=device)

    # The first calls on freshly pinned host buffers run slow (one-time mapping of the pages for
    # the copy engines: up to ~4x the steady state), so the warm-up is at least five calls.
    for _ in range(max(5, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, min(args.steps, 10))
    barrier(dist, device)
    s_ev.record(stream)
    for _ in range(steps):
        step()
    e_ev.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    ms = max_over_ranks(dist, s_ev.elapsed_time(e_ev), device)
    fl = step_flops(case)
    val = aggregate_tflops(world, fl["fwd"] + fl["bwd"], steps, ms)
    swa.swa_check_device(device)
    return {"value": val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms / steps, "steps": steps, "units_per_chunk": U,
            "api": "swa_attn_fwd_bwd_host"}


def _layer_calls(swa, inp, W: int, scale: float, causal: bool = True):
    """Forward and backward calls of one layer on preallocated outputs and workspace, so that a
    timed repetition launches the kernels and allocates nothing."""
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    dev = q.device
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if q.dtype == torch.float32:
        nws = swa.swa_attn_f32_workspace_bytes(B, Hq, Hkv, Lq, Lk, D)
    else:
        nws = swa.swa_attn_bwd_workspace_bytes(B, Hq, Lq, D)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    fwd_ws = ws if q.dtype == torch.float32 else None

    def fwd():
        swa.swa_attn_fwd(q, k, v, W, scale, out=o, lse=lse, causal=causal, workspace=fwd_ws)

    def bwd():
        swa.swa_attn_bwd(q, k, v, o, do, lse, W, scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                         causal=causal)

    return fwd, bwd


def measure_other_workloads(swa, device) -> dict:
    """Full-causal GQA layer (fwd and bwd timed separately), the headline layer in fp16, fp32, with
    64- and 256-wide heads, a query suffix and a two-sided window over the headline keys, and the
    12-layer mixed step with its peak memory.  Outputs and workspaces are allocated before timing."""
    res = {}
    stream = torch.cuda.current_stream(device)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / reps

    def layer(name, what, case, dtype=torch.bfloat16, Lq=None, causal=True, both=True):
        inp = si.make_inputs(case, device=str(device), dtype=dtype)
        if Lq is not None:
            for key in ("q", "do"):
                inp[key] = inp[key][:, :, case.N - Lq:].contiguous()
        Lq = case.N if Lq is None else Lq
        pairs = window_pairs(Lq, case.N, case.W, causal) * case.B * case.Hq
        fwd, bwd = _layer_calls(swa, inp, case.W, case.softmax_scale, causal)
        f_ms = timed(fwd)
        b_ms = timed(bwd)
        r = {"workload": what, "fwd_ms": f_ms, "bwd_ms": b_ms,
             "fwd_tflops": 4 * case.D * pairs / (f_ms * 1e-3) / 1e12,
             "bwd_tflops": 10 * case.D * pairs / (b_ms * 1e-3) / 1e12}
        if both:
            r["fwd_bwd_tflops"] = 14 * case.D * pairs / ((f_ms + b_ms) * 1e-3) / 1e12
        if Lq != case.N or not causal:
            r["pairs_per_head"] = pairs // (case.B * case.Hq)
        res[name] = r
        del inp, fwd, bwd
        torch.cuda.empty_cache()

    layer("gqa_causal_8k", "B=1 Hq=32 Hkv=8 N=8192 D=128 full causal", si.gqa_causal_case(),
          both=False)
    long32 = si.long_swa_case(32768)
    layer("long_swa_fp16", "B=1 Hq=32 Hkv=16 N=32768 D=128 W=1024, fp16 tensors", long32,
          dtype=torch.float16)
    layer("long_swa_d64", "B=1 Hq=32 Hkv=16 N=32768 D=64 W=1024",
          dataclasses.replace(long32, D=64))
    layer("long_swa_d256", "B=1 Hq=32 Hkv=16 N=32768 D=256 W=1024",
          dataclasses.replace(long32, D=256))
    layer("long_swa_fp32", "B=1 Hq=32 Hkv=16 N=32768 D=128 W=1024, fp32 tensors", long32,
          dtype=torch.float32)
    layer("suffix_queries_8k_of_32k", "B=1 Hq=32 Hkv=16 Lq=8192 Lk=32768 D=128 W=1024 causal, "
          "queries = the last 8192 key positions", long32, Lq=8192)
    layer("twosided_32k", "B=1 Hq=32 Hkv=16 N=32768 D=128 W=1024 two-sided (|i - j| < W)", long32,
          causal=False)
    res["mixed_12_layers"] = measure_mixed_step(swa, device, timed)
    return res


def measure_mixed_step(swa, device, timed) -> dict:
    """The 12-layer mixed step (layers 5 and 11 full causal, the rest W = 1024; N = 30,553): the
    forward of every layer (O and LSE kept), then the backward from layer 11 down to 0.  Each layer
    has its own inputs, O and LSE; the layers' gradients share one set of buffers, as a training
    step hands each layer's gradients on before the next backward.  Peak memory is the most torch
    held during the step, with and without the inputs."""
    layers = si.mixed_layer_cases()
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(device)
    before = torch.cuda.memory_allocated(device)
    data = [si.make_inputs(c, device=str(device)) for c in layers]
    torch.cuda.synchronize(device)
    inputs_bytes = torch.cuda.memory_allocated(device) - before
    c0 = layers[0]
    outs = [(torch.empty_like(d["q"]),
             torch.empty((c0.B, c0.Hq, c0.N), dtype=torch.float32, device=device)) for d in data]
    dq, dk, dv = (torch.empty_like(data[0]["q"]), torch.empty_like(data[0]["k"]),
                  torch.empty_like(data[0]["v"]))
    ws = torch.empty(swa.swa_attn_bwd_workspace_bytes(c0.B, c0.Hq, c0.N, c0.D),
                     dtype=torch.uint8, device=device)

    def mixed_step():
        for i, c in enumerate(layers):
            swa.swa_attn_fwd(data[i]["q"], data[i]["k"], data[i]["v"], c.W, c.softmax_scale,
                             out=outs[i][0], lse=outs[i][1])
        for i in reversed(range(len(layers))):
            c = layers[i]
            swa.swa_attn_bwd(data[i]["q"], data[i]["k"], data[i]["v"], outs[i][0], data[i]["do"],
                             outs[i][1], c.W, c.softmax_scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    m_ms = timed(mixed_step, reps=3)
    torch.cuda.synchronize(device)
    peak = torch.cuda.max_memory_allocated(device) - before
    tot = sum(step_flops(c)["fwd"] + step_flops(c)["bwd"] for c in layers)
    res = {
        "workload": "12 layers (W=1024 except layers 5 and 11 full causal), B=1 Hq=32 Hkv=16 "
                    "N=30553 D=128, fwd all then bwd 11..0",
        "step_ms": m_ms,
        "tflops": tot / (m_ms * 1e-3) / 1e12,
        "peak_gb": peak / 1e9,
        "peak_gb_above_inputs": (peak - inputs_bytes) / 1e9,
        "inputs_gb": inputs_bytes / 1e9,
    }
    del data, outs, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------------------------
# Reference arm: the fp64 oracle on the host cores
# ------------------------------------------------------------------------------------------------

def run_reference(args, world, rank, local):
    """The fp64 oracle on the host cores, on the headline workload: each step is a bounded sample
    of it (`--ref-rows` mid-sequence query rows of one query head, forward + backward), and the
    value counts the window-effective flops of the sampled rows."""
    if rank != 0:
        return
    case = si.long_swa_case(32768)
    R = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(case, rows_per_sample=R, samples=1)
    t0 = time.perf_counter()
    smp = oracle_sample(case, rows_per_sample=R, samples=args.steps)
    dt = time.perf_counter() - t0
    val = smp["value"]
    result = {
        "impl": "reference",
        "metric": METRIC,
        "value": val,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(case, world),
        "cpu_baseline": {
            "value": val, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{args.steps} steps x {R} query rows (mid-sequence) of one head of the "
                      "workload, fp64 NumPy oracle fwd + bwd",
            "cpu_model": cpu_model(), "cpu_count": os.cpu_count(),
        },
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(result), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--bwd", choices=("fused", "split"), default="split",
                    help="backward path of the timed step (the other is timed after it)")
    ap.add_argument("--no-memory", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-soak", action="store_true",
                    help="skip the untimed clock soak after the timed region (profiler runs)")
    ap.add_argument("--seq-len", type=int, default=32768,
                    help="sequence length of the timed layer (profiler runs on a smaller layer; "
                         "the headline is 32768)")
    ap.add_argument("--head-dim", type=int, choices=(64, 128, 256), default=128,
                    help="head dimension of the timed layer (profiler runs; the headline is 128)")
    ap.add_argument("--ref-rows", type=int, default=256,
                    help="query rows per step of the reference arm's oracle sample")
    ap.add_argument("--cpu-rows", type=int, default=2048,
                    help="query rows per head in the oracle's row samples of the long layers")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
