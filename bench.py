"""Benchmark of the fused local MoE forward on the fine-grained headline workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME] [--dtype f16] [--l2-flush] [--no-cpu-baseline]

One step = one moe_forward (route -> dispatch -> grouped gate/up + SwiGLU ->
grouped down with weighted un-permute -> combine) over T tokens whose inputs
are already resident in HBM.  Prints ONE JSON line (rank 0).  Under torchrun
each rank runs the same workload on its own GPU (tokens are independent, so
ranks need no data exchange: weak scaling); the time is the max over ranks.

Exactly K steps are timed between a barrier and device synchronisations; when
K steps take less than --min-seconds (0.5 s), that timed loop is repeated so
that the nvidia-smi sampler (50 ms) records at least ~10 clock samples inside
the window.  There are at least two repetitions: the step time is the mean
over all but the last, which also records the per-stage events (an event
between two launches stops their programmatic-launch overlap) and gives the
stage times and the roofline.  The roofline's peak follows the window's clock
record: the burst BF16 figure when the median SM clock sat at its maximum with
no sw_power_cap sample, else the sustained one.  The default run then measures the other four workloads and
the headline in FP16 the same way, under the line's "workloads" key.

``--impl reference`` times the FP64 CPU oracle (the only reference this
method has) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "MoE fwd tokens/s; grouped-GEMM TFLOP/s as % of GB300 BF16 peak (1 GPU)"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "finegrained_bf16"
def launches_per_step(T: int, E: int) -> int:
    """Kernels of one fused forward: route, count, [scan], scatter, gather,
    gate/up GEMM, down GEMM, combine.  The scan kernel runs only when the
    chunk histogram table (256-token chunks x (E+1) words) exceeds 16384
    words; below that the scatter blocks scan it themselves."""
    chunks = (T + 255) // 256
    return 7 + (1 if chunks * (E + 1) > 16384 else 0)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per grouped_gemm_tc launch (mean of the gate/up and the down
# launch, dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of
# each workload, with the SHA-256 of the kernel source's code (comments and
# white space left out) it was taken on; it is reported as null once that
# code changes.
GEMM_TRAFFIC = {
    # ncu --set full, one launch each on the headline workload: gate/up reads
    # 1.141058 GB and writes 265.725696 MB, down reads 0.646926 GB and writes
    # 373.762816 MB (ncu's units; the GB figures are rounded to the kilobyte)
    "finegrained_bf16": {"bytes_per_launch": (1141058000 + 265725696 + 646926000 + 373762816) / 2,
                         "code_sha256": "e15a00f4548dfbd7a723e0d81565253554c1d21e59cb26ec407440f0a3802ee4"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--mode", choices=["forward", "backward"], default="forward",
                   help="backward: time the first-order training backward chain instead")
    p.add_argument("--bwd-strategy", choices=["scalar", "auto", "tensor_core"], default="auto",
                   help="expert backward strategy of --mode backward")
    p.add_argument("--routing", choices=["softmax", "sigmoid"], default="softmax",
                   help="sigmoid: time the fused forward with sigmoid group-limited routing "
                        "(groups of 8 experts, half the groups kept, top-two group score, "
                        "renormalised, scale 2.5)")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--dtype", choices=["bf16", "f16"], default=None,
                   help="store the workload in this dtype instead of its own")
    p.add_argument("--tokens", type=int, default=None,
                   help="override the workload's token count (small cases for profiler captures)")
    p.add_argument("--e2e-steps", type=int, default=None,
                   help="steps of the host-buffer legs (default: the device loop's steps x repeats, so "
                        "that they run as long and see the same clocks)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="skip the extra measurement of the step replayed from a captured CUDA graph")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other workloads measured after the headline in the default run")
    p.add_argument("--min-seconds", type=float, default=0.5,
                   help="repeat the K timed steps until this much timed work (clock samples >= 10)")
    p.add_argument("--side-steps", type=int, default=20, help="timed steps per repetition, other workloads")
    p.add_argument("--side-seconds", type=float, default=0.5, help="--min-seconds of the other workloads")
    p.add_argument("--l2-flush", action="store_true",
                   help="write a 256 MB buffer before every step (outside the forward's events); "
                        "the per-step time is then the forward's own event span")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target wall time of the oracle sample")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def bench_workload(args):
    import dataclasses
    from top_routing_grouped_fp32_gb300.inputs import WORKLOADS, with_dtype
    wl = with_dtype(WORKLOADS[args.workload], args.dtype or WORKLOADS[args.workload].dtype)
    if args.tokens is not None:
        wl = dataclasses.replace(wl, name=f"{wl.name}_T{args.tokens}", T=args.tokens)
    return wl


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def code_sha256(rel: str) -> str:
    """SHA-256 of a C/C++/CUDA source with its comments removed and every run
    of white space collapsed to one blank: editing a comment leaves it
    unchanged, editing code does not.  String and character literals are
    copied as they stand."""
    with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
        text = f.read()
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    code = " ".join("".join(out).split())
    return hashlib.sha256(code.encode()).hexdigest()


class ClockSampler:
    """nvidia-smi clock / power / throttle sampling; only samples whose
    timestamps fall inside the timed window are summarised."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float):
        """Summary of the samples taken between wall-clock times t0 and t1."""
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in text.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                v_sm, v_max, v_pw = float(parts[2]), float(parts[3]), float(parts[4])
            except ValueError:
                continue
            if not (t0 <= ts <= t1):
                continue
            sm.append(v_sm)
            smax.append(v_max)
            power.append(v_pw)
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU baseline / reference arm: the FP64 oracle on the host cores
# --------------------------------------------------------------------------

def _host_inputs(wl):
    """The workload's inputs as stored bits on the host (drawn on the GPU when
    one is present, so they are the same bits the native arm uses)."""
    import torch
    from top_routing_grouped_fp32_gb300.inputs import make_inputs, to_stored_numpy
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(wl, device=dev)
    out = {k: to_stored_numpy(inp[k]) for k in ("x", "logits", "gate", "up", "down")}
    del inp
    if dev == "cuda":
        torch.cuda.empty_cache()
    return out


def oracle_sample_rate(wl, host, target_s: float, tokens_offset: int = 0):
    """Times oracle.forward_tokens (route + k experts + weighted sum per token,
    FP64, OpenMP over tokens) on a token sample sized to about target_s
    seconds.  Returns (tokens/s, tokens, seconds, threads)."""
    import numpy as np
    import oracle
    oracle.build()
    threads = oracle.num_threads()

    def run(n):
        toks = (np.arange(n) * 7919 + tokens_offset) % wl.T
        t0 = time.perf_counter()
        oracle.forward_tokens(host["x"], host["logits"], host["gate"], host["up"], host["down"],
                              wl.dtype, wl.dtype, wl.top_k, wl.renormalize, toks)
        return time.perf_counter() - t0

    n = max(threads, 8)
    dt = run(n)
    n = int(min(wl.T, max(n, n * target_s / max(dt, 1e-3))))
    dt = run(n)
    return n / dt, n, dt, threads


def run_reference(args, rank, world):
    """The reference arm: the oracle as it stands, timed per step on a bounded
    sample of the workload's tokens."""
    import numpy as np
    import oracle
    from top_routing_grouped_fp32_gb300.inputs import WORKLOADS
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    host = _host_inputs(wl)
    oracle.build()
    threads = oracle.num_threads()
    # size one step's sample so that warm-up + steps take about three minutes
    rate, _, _, _ = oracle_sample_rate(wl, host, target_s=2.0)
    budget = 180.0 / max(1, args.steps + args.warmup)
    per_step = int(max(threads, min(wl.T, rate * budget)))

    def step(i):
        toks = (np.arange(per_step) * 7919 + i * per_step) % wl.T
        oracle.forward_tokens(host["x"], host["logits"], host["gate"], host["up"], host["down"],
                              wl.dtype, wl.dtype, wl.top_k, wl.renormalize, toks)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    sample = (f"{per_step} tokens per step of {wl.name} through the FP64 oracle "
              f"(route + {wl.top_k} SwiGLU experts + weighted sum per token)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, l2_flush=False):
    s = 4 if wl.dtype == "f32" else 2
    if l2_flush:
        l2 = "flushed: a 256 MB buffer is written before every step (outside the timed events)"
    else:
        l2 = ("no flush: every step streams all expert weights "
              f"({3 * wl.E * wl.H * wl.I * s / 1e9:.3g} GB) and the dispatched rows; above the "
              "129 MB L2 for every workload but the tiny one, which is launch-bound")
    return {"workload": wl.name, "T": wl.T, "E": wl.E, "top_k": wl.top_k, "H": wl.H, "I": wl.I,
            "renormalize": wl.renormalize, "seed": wl.seed, "weights_dtype": wl.dtype, "l2": l2}


# --------------------------------------------------------------------------
# native arm
# --------------------------------------------------------------------------

# workloads measured after the headline in the default run, each a few hundred
# milliseconds: (workload, dtype override)
SIDE_WORKLOADS = [("mixtral_bf16", None), ("skewed_bf16", None), ("decode_bf16", None),
                  ("tiny_fp32", None), ("finegrained_bf16", "f16")]
STAGES = ["route", "dispatch", "gate_up_gemm", "down_gemm", "combine"]
L2_FLUSH_BYTES = 256 << 20


def tensor_peak(peaks, src, clocks):
    """The BF16 tensor peak that matches the timed window's own clock record:
    the burst figure when the median SM clock sat at its maximum and no
    sw_power_cap sample fell inside the window (or no record exists), else the
    sustained figure measured under the power cap."""
    burst = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", burst))
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in clocks.get("reasons", [])
    if sm is None or smax is None:
        return burst, f"{src} bf16_tflops (burst; no clock record for the window)"
    if sm >= smax - 15 and not capped:
        return burst, f"{src} bf16_tflops (burst: median SM clock {sm:.0f} of {smax:.0f} MHz, no sw_power_cap)"
    why = "sw_power_cap active" if capped else "clock below max"
    return sus, (f"{src} bf16_tflops_sustained (median SM clock {sm:.0f} of {smax:.0f} MHz, {why})")


def roofline_for(wl, stage, touched, clocks, peaks, peaks_src, traffic=None):
    """Roofline of the dominant kernel, grouped_gemm_tc (its two launches per
    step: gate/up + SwiGLU and down + weighted un-permute).  Tensor-bound
    workloads: 6*N*H*I FLOP over the two launches' summed time against the BF16
    peak that the clock record selects.  The decode workload streams weights:
    the touched experts' 3*H*I weights over the same time against the measured
    copy bandwidth.  FP32 experts run on the FFMA pipe: against 152 SMs x 128
    lanes x 2 FLOP x the max SM clock."""
    N = wl.T * wl.top_k
    t_gu, t_dn = stage["gate_up_gemm"], stage["down_gemm"]
    gemm_s = (t_gu + t_dn) * 1e-3
    flops = 6.0 * N * wl.H * wl.I
    s_el = 4 if wl.dtype == "f32" else 2
    wbytes = touched * 3.0 * wl.H * wl.I * s_el
    hbm = float(peaks["hbm_gbs"])
    if wl.dtype == "f32":
        smax = clocks.get("sm_max_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
        peak = 152 * 128 * 2 * smax * 1e6 / 1e12
        ach = flops / gemm_s / 1e12
        return {"bound": "alu", "kernel": "grouped_gemm_simt (FP32 FFMA, gate/up + down)", "achieved": ach,
                "peak": peak, "unit": "TFLOP/s", "frac": ach / peak, "traffic": None,
                "peak_source": f"152 SMs x 128 FP32 lanes x 2 FLOP x {smax:.0f} MHz",
                "algorithmic_per_launch": f"6*N*H*I / 2 launches = {flops / 2:.4e} FLOP"}
    if wl.name.startswith("decode"):
        ach = wbytes / gemm_s / 1e9
        return {"bound": "hbm", "kernel": "grouped_gemm_tc (gate/up + SwiGLU, down + weighted un-permute)",
                "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": traffic,
                "peak_source": f"{peaks_src} hbm_gbs",
                "algorithmic_per_launch": (f"touched experts' weights 3*H*I*2 x {touched} / 2 launches = "
                                           f"{wbytes / 2:.4e} B"),
                "gate_up_only": {"achieved": touched * 2.0 * wl.H * wl.I * s_el / (t_gu * 1e-3) / 1e9,
                                 "unit": "GB/s"}}
    peak, psrc = tensor_peak(peaks, peaks_src, clocks)
    burst = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", burst))
    ach = flops / gemm_s / 1e12
    gu = 4.0 * N * wl.H * wl.I / (t_gu * 1e-3) / 1e12
    dn = 2.0 * N * wl.H * wl.I / (t_dn * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": "grouped_gemm_tc (gate/up + SwiGLU, down + weighted un-permute)",
            "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak, "traffic": traffic,
            "peak_source": psrc, "frac_of_burst": ach / burst, "frac_of_sustained": ach / sus,
            "algorithmic_per_launch": f"6*N*H*I / 2 launches = {flops / 2:.4e} FLOP",
            "gate_up": {"achieved": gu, "frac": gu / peak, "flop": 4.0 * N * wl.H * wl.I},
            "down": {"achieved": dn, "frac": dn / peak, "flop": 2.0 * N * wl.H * wl.I}}


def gemm_traffic(wl):
    """Mean DRAM bytes per grouped_gemm_tc launch from the committed ncu capture
    of this workload, or None once the kernel source has changed."""
    rec = GEMM_TRAFFIC.get(wl.name)
    if not rec or rec["code_sha256"] != code_sha256("top_routing_grouped_fp32_gb300/csrc/gemm_tc.cu"):
        return None
    return rec["bytes_per_launch"]


def measure_forward(moe, wl, args, world, dev, min_seconds, K, warmup, keep=False):
    """Warm-up, then repetitions of exactly K timed forward steps (each between
    a barrier and device synchronisations, events on the launching stream)
    until at least `min_seconds` of timed work, so that the clock sampler sees
    at least ~10 samples inside the window.  The step time is the mean over
    the plain repetitions; the last repetition also records events between
    the launches, and the per-stage times (so the roofline) come from it, under
    the same clocks."""
    import torch
    from top_routing_grouped_fp32_gb300.inputs import make_inputs
    inp = make_inputs(wl, device=dev)
    experts = moe.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    ws = experts.forward_workspace(wl.T, wl.top_k, inp["logits"].dtype)
    y = torch.empty((wl.T, wl.H), dtype=inp["x"].dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if args.l2_flush else None

    def step(events=None, i=0):
        if flush is not None:
            flush.fill_(i & 0xFF)  # 256 MB written: nothing of the last step stays in the 129 MB L2
        experts.forward(inp["x"], inp["logits"], wl.top_k, wl.renormalize, y=y, workspace=ws,
                        stream=stream, events=events)

    for i in range(max(3, warmup)):
        step(i=i)
    torch.cuda.synchronize(dev)
    assert moe.moe_get_device_status(ws) == 0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in [x for row in ev for x in row]:
        e.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize(dev)

    stage_sum = {n: 0.0 for n in STAGES}
    span_sum = 0.0  # route start -> combine end, summed over instrumented steps (flush excluded)
    rep_ms = []
    inst_reps = []
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    w0 = time.time()
    reps = 2
    r = 0
    while r < reps:
        # Stage events between launches stop the programmatic-launch overlap of
        # the kernels they separate, so only the last repetition (every one
        # under --l2-flush, whose step time is the event span) records them;
        # the others time K plain steps.
        inst = flush is not None or r == reps - 1
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for i in range(K):
            step(ev[i] if inst else None, i)
        end.record(stream)
        torch.cuda.synchronize(dev)
        rep_ms.append(max_over_ranks(start.elapsed_time(end), world, dev))
        inst_reps.append(inst)
        if inst:
            for i in range(K):
                for j, n in enumerate(STAGES):
                    stage_sum[n] += ev[i][j].elapsed_time(ev[i][j + 1])
                span_sum += ev[i][0].elapsed_time(ev[i][5])
        if r == 0:  # the same repetition count on every rank; at least one plain and one instrumented
            reps = max(2, int(math.ceil(min_seconds * 1e3 / max(rep_ms[0], 1e-3))))
            reps = int(max_over_ranks(float(reps), world, dev))
        r += 1
    w1 = time.time()
    clock_info = clocks.stop(w0, w1)
    status = moe.moe_get_device_status(ws)
    n_inst = K * sum(inst_reps)
    stage = {n: v / n_inst for n, v in stage_sum.items()}
    if flush is not None:
        # the flush is outside the forward: the per-step time is its event span
        ms_step = max_over_ranks(span_sum / n_inst, world, dev)
        steps = K * reps
    else:
        plain = [m for m, i in zip(rep_ms, inst_reps) if not i]
        steps = K * len(plain)
        ms_step = sum(plain) / steps
    lay = experts.forward_layout(wl.T, wl.top_k, inp["logits"].dtype)
    off = ws[lay["offsets"]:lay["offsets"] + 4 * (wl.E + 1)].view(torch.int32).cpu()
    touched = int(((off[1:] - off[:-1]) != 0).sum().item())
    res = {"value": wl.T * world / (ms_step * 1e-3), "ms_per_step": ms_step, "repeats": reps,
           "rep_ms_per_step": [m / K for m in rep_ms], "rep_stage_events": inst_reps,
           "stages_ms": stage, "clocks": clock_info, "touched": touched, "device_status": status,
           "gpu_launches": launches_per_step(wl.T, wl.E) * steps}
    if not args.no_graph and flush is None:
        res["graph"] = measure_graph(experts, inp, wl, y, ws, stream, K, steps, world, dev)
    if keep:
        res["_state"] = (inp, experts, ws, y, stream)
    else:
        del inp, experts, ws, y, flush
        torch.cuda.empty_cache()
    return res


def measure_graph(experts, inp, wl, y, ws, stream, K, steps, world, dev):
    """The same step captured once into a CUDA graph (the library's calls only
    enqueue work, so they capture) and replayed: as many replays as the plain
    timed steps, K per event pair.  An extra figure beside the call a user
    makes; it shows how much of a launch-bound step is host work."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        experts.forward(inp["x"], inp["logits"], wl.top_k, wl.renormalize, y=y, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total, done = 0.0, 0
    while done < steps:
        n = min(K, steps - done)
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for _ in range(n):
            g.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        total += max_over_ranks(start.elapsed_time(end), world, dev)
        done += n
    ms = total / done
    del g
    return {"value": wl.T * world / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": done,
            "what": "the step replayed from one captured CUDA graph"}


def measure_e2e(wl, world, dev, inp, experts, stream, Ke):
    """End to end through the host-buffer entry points: every step copies its
    inputs in from pinned host memory and its result out, inside the timed
    region.  `e2e` is the pipelined entry point (moe_host_pipeline_*, the
    copies of neighbouring steps overlap the forward between them; two sets of
    host buffers alternate); `e2e_serial` is one moe_forward_host call per
    step (copy in, forward, copy out on one stream).  Host wall clock between
    two device synchronisations."""
    import torch
    xh = [inp["x"].cpu().pin_memory() for _ in range(2)]
    lh = [inp["logits"].cpu().pin_memory() for _ in range(2)]
    yh = [torch.empty((wl.T, wl.H), dtype=inp["x"].dtype).pin_memory() for _ in range(2)]
    pipe = experts.host_pipeline(wl.T, wl.top_k, wl.renormalize, logits_dtype=inp["logits"].dtype,
                                 depth=2, stream=stream)
    for i in range(3):
        pipe.submit(xh[i % 2], lh[i % 2], yh[i % 2])
    pipe.sync()
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(Ke):
        pipe.submit(xh[i % 2], lh[i % 2], yh[i % 2])
    pipe.sync()
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
    pipe.close()
    wsh = experts.forward_host_workspace(wl.T, wl.top_k, inp["logits"].dtype)
    for _ in range(3):
        experts.forward_host(xh[0], lh[0], wl.top_k, wl.renormalize, yh[0], wsh, stream=stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(Ke):
        experts.forward_host(xh[0], lh[0], wl.top_k, wl.renormalize, yh[0], wsh, stream=stream)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
    h2d = xh[0].numel() * xh[0].element_size() + lh[0].numel() * lh[0].element_size()
    d2h = yh[0].numel() * yh[0].element_size()
    del wsh
    return ({"value": wl.T * world * Ke / (e2e_ms * 1e-3), "unit": UNIT,
             "api": "moe_host_pipeline_submit (depth 2), one call per step",
             "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            {"value": wl.T * world * Ke / (e2e_serial_ms * 1e-3), "unit": UNIT,
             "api": "moe_forward_host, one call per step"})


def run_native(args, rank, world, local):
    import torch
    import top_routing_grouped_fp32_gb300 as moe
    from top_routing_grouped_fp32_gb300.inputs import WORKLOADS, with_dtype

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the native arm has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    moe.load()
    wl = bench_workload(args)
    K = args.steps
    res = measure_forward(moe, wl, args, world, dev, args.min_seconds, K, args.warmup, keep=True)
    inp, experts, ws, y, stream = res.pop("_state")
    assert inp["x"].dtype == {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[wl.dtype]
    Ke = max(1, args.e2e_steps if args.e2e_steps is not None else K * res["repeats"])
    e2e, e2e_serial = measure_e2e(wl, world, dev, inp, experts, stream, Ke)
    del inp, experts, ws, y
    torch.cuda.empty_cache()
    peaks, peaks_src = load_peaks()

    line = None
    if rank == 0:
        roof = roofline_for(wl, res["stages_ms"], res["touched"], res["clocks"], peaks, peaks_src,
                            gemm_traffic(wl))
        line = {
            "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "repeats": res["repeats"],
            "rep_ms_per_step": res["rep_ms_per_step"], "rep_stage_events": res["rep_stage_events"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded randn, BF16 weights ~N(0,1/fan_in)); no dataset, random-init weights",
            "config": workload_config(wl, args.l2_flush),
            "stages_ms": res["stages_ms"],
            "roofline": roof,
            "e2e": e2e, "e2e_serial": e2e_serial,
            "gpu_launches": res["gpu_launches"], "graph": res.get("graph"),
            "clocks": res["clocks"],
            "device_status": res["device_status"],
        }
    # the other workloads (and the headline in FP16), a few hundred ms each
    if args.workload == DEFAULT_WORKLOAD and args.tokens is None and args.dtype is None \
            and not args.no_workloads:
        side = {}
        for name, dt in SIDE_WORKLOADS:
            swl = with_dtype(WORKLOADS[name], dt or WORKLOADS[name].dtype)
            key = swl.name
            r = measure_forward(moe, swl, args, world, dev, args.side_seconds, args.side_steps, 5)
            if rank == 0:
                side[key] = {"config": workload_config(swl, args.l2_flush), "value": r["value"], "unit": UNIT,
                             "ms_per_step": r["ms_per_step"], "steps": args.side_steps,
                             "repeats": r["repeats"], "stages_ms": r["stages_ms"],
                             "roofline": roofline_for(swl, r["stages_ms"], r["touched"], r["clocks"],
                                                      peaks, peaks_src, gemm_traffic(swl)),
                             "touched_experts": r["touched"], "clocks": r["clocks"], "graph": r.get("graph"),
                             "device_status": r["device_status"]}
        if rank == 0:
            line["workloads"] = side
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = _host_inputs(wl)
        rate, n, dt, threads = oracle_sample_rate(wl, host, args.cpu_seconds)
        # the same oracle on one thread, on a smaller sample (a few seconds)
        import oracle
        oracle.set_threads(1)
        rate1, n1, dt1, _ = oracle_sample_rate(wl, host, min(5.0, args.cpu_seconds / 3))
        oracle.set_threads(threads)
        line["cpu_baseline"] = {
            "value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": (f"{n} tokens of {wl.name} through the FP64 oracle (route + {wl.top_k} SwiGLU "
                       f"experts + weighted sum per token) in {dt:.1f} s"),
            "value_1thread": rate1,
            "sample_1thread": f"{n1} tokens in {dt1:.1f} s on one thread"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_backward(args, rank, world, local):
    """Times the first-order backward chain (user guide section 12) after a
    staged forward: combine backward -> expert backward -> dispatch backward
    -> router backward.  The step time is K plain steps timed in blocks; K more
    steps, in blocks alternating with those, record events between the stages
    for the split.  The expert
    backward's roofline is the tensor pipe (measured bf16 peak) for the
    tensor-core strategy, else the FP32 FMA pipe: 152 SMs x 128 lanes x 2 FLOP
    x the max SM clock."""
    import torch
    import top_routing_grouped_fp32_gb300 as moe
    from top_routing_grouped_fp32_gb300.inputs import WORKLOADS, make_inputs, with_dtype
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = bench_workload(args)
    inp = make_inputs(wl, device=dev)
    ex = moe.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, w = moe.moe_route(inp["logits"], wl.top_k, wl.renormalize)
    d = moe.moe_dispatch(idx, wl.E, x=inp["x"])
    eo = ex.forward_dispatched(d.x_disp, d.offsets)
    g = torch.Generator(device=dev).manual_seed(99)
    dy = torch.randn((wl.T, wl.H), generator=g, device=dev).to(inp["x"].dtype)
    N = wl.T * wl.top_k
    bws = moe._workspace(ex._lib.moe_experts_backward_workspace_size(ex.handle, N), dev)

    def step(ev=None):
        rec = (lambda j: ev[j].record()) if ev else (lambda j: None)
        rec(0)
        dex, dwt = moe.moe_combine_backward(eo, d.perm, w, dy, wl.top_k)
        rec(1)
        dinput, dgate, dup, ddown = ex.backward(d.x_disp, d.offsets, dex, workspace=bws,
                                                strategy=args.bwd_strategy)
        rec(2)
        moe.moe_dispatch_backward(dinput, d.perm, wl.T, wl.top_k)
        rec(3)
        moe.moe_router_backward(inp["logits"], idx, dwt, "softmax", wl.renormalize, 1.0)
        rec(4)

    K = max(1, args.steps)
    W = max(3, args.warmup)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    w0 = time.time()
    # K plain steps give the step time; K more with events between the stages
    # (which stop the overlap of the launches they separate) give the split.
    # The two kinds alternate in blocks, so that both see the same clocks.
    nblk = min(5, K)
    plain_ms, plain_steps, done = 0.0, 0, 0
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for b in range(nblk):
        n = (K - done) // (nblk - b)
        torch.cuda.synchronize(dev)
        start.record()
        for _ in range(n):
            step()
        end.record()
        torch.cuda.synchronize(dev)
        plain_ms += start.elapsed_time(end)
        plain_steps += n
        for i in range(done, done + n):
            step(evs[i])
        done += n
    torch.cuda.synchronize(dev)
    total = plain_ms / plain_steps
    clock_info = clocks.stop(w0, time.time())
    names = ["combine_backward", "experts_backward", "dispatch_backward", "router_backward"]
    st = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
          for j, n in enumerate(names)}
    flops = 16.0 * N * wl.H * wl.I  # recompute g,u (4) + da (2) + dinput (4) + 3 weight grads (6)
    ach = flops / (st["experts_backward"] * 1e-3) / 1e12
    tensor = args.bwd_strategy == "tensor_core" or (args.bwd_strategy == "auto" and wl.dtype != "f32")
    if tensor:
        peaks, peaks_src = load_peaks()
        peak, psrc = tensor_peak(peaks, peaks_src, clock_info)
        sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
        roof = {"bound": "tensor", "kernel": "experts backward (tcgen05 chain)", "achieved": ach,
                "peak": peak, "unit": "TFLOP/s", "frac": ach / peak, "peak_source": psrc,
                "frac_of_burst": ach / float(peaks["bf16_tflops"]), "frac_of_sustained": ach / sus}
    else:
        peak = 152 * 128 * 2 * 2.07e9 / 1e12
        roof = {"bound": "alu", "kernel": "experts backward (FP32 FMA)", "achieved": ach,
                "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "peak_source": "152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz"}
    roof["algorithmic_per_launch"] = f"16*N*H*I = {flops:.4e} FLOP"
    line = {"metric": "MoE first-order backward tokens/s", "value": wl.T / (total * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": W, "mode": "backward",
            "bwd_strategy": "tensor_core" if tensor else "scalar",
            "ms_per_step": total, "higher_is_better": True, "dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl), "stages_ms": st, "roofline": roof, "clocks": clock_info}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_sigmoid(args, rank, world, local):
    """The fused forward with sigmoid group-limited routing (user guide section
    10) on the workload's shapes; one event pair around the timed steps, and
    the routing kernel timed on its own."""
    import torch
    import top_routing_grouped_fp32_gb300 as moe
    from top_routing_grouped_fp32_gb300.inputs import make_inputs
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = bench_workload(args)
    inp = make_inputs(wl, device=dev)
    ex = moe.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    groups = max(1, wl.E // 8)
    opts = dict(groups=groups, selected_groups=max(1, groups // 2), group_top_two=wl.E // groups >= 2,
                renormalize=True, scale=2.5)
    y = torch.empty((wl.T, wl.H), dtype=inp["x"].dtype, device=dev)
    ws = ex.forward_workspace(wl.T, wl.top_k, inp["logits"].dtype)

    def step():
        ex.forward_sigmoid_grouped(inp["x"], inp["logits"], wl.top_k, y=y, workspace=ws, **opts)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    w0 = time.time()
    e0.record()
    for _ in range(K):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop(w0, time.time())
    ms = e0.elapsed_time(e1) / K
    # the routing kernel alone: outputs allocated once and the C ABI called
    # directly, so that the loop is not bound by per-call host work
    from top_routing_grouped_fp32_gb300 import _lib
    lib = moe.load()
    ridx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    rw = torch.empty((wl.T, wl.top_k), dtype=inp["logits"].dtype, device=dev)
    ropt = moe.group_options(wl.top_k, opts["groups"], opts["selected_groups"], opts["group_top_two"],
                             opts["renormalize"], opts["scale"])
    rargs = (inp["logits"].data_ptr(), moe._code(inp["logits"]), wl.T, wl.E, None, ctypes.byref(ropt),
             ridx.data_ptr(), rw.data_ptr(), None, torch.cuda.current_stream(dev).cuda_stream)
    for _ in range(3):
        _lib.check(lib.moe_route_sigmoid_grouped(*rargs))
    torch.cuda.synchronize(dev)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record()
    for _ in range(K):
        lib.moe_route_sigmoid_grouped(*rargs)
    r1.record()
    torch.cuda.synchronize(dev)
    route_ms = r0.elapsed_time(r1) / K
    peaks, peaks_src = load_peaks()
    sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    N = wl.T * wl.top_k
    ach = 6.0 * N * wl.H * wl.I / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": wl.T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "routing": "sigmoid",
            "routing_options": opts, "dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl), "route_sigmoid_ms": route_ms,
            "roofline": {"bound": "tensor", "kernel": "whole fused forward (per-kernel split not instrumented)",
                         "achieved": ach, "peak": sus, "unit": "TFLOP/s", "frac": ach / sus,
                         "peak_source": f"{peaks_src} bf16_tflops_sustained",
                         "algorithmic_per_step": f"6*N*H*I = {6.0 * N * wl.H * wl.I:.4e} FLOP"},
            "clocks": clock_info, "device_status": moe.moe_get_device_status(ws)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.mode == "backward":
        return run_backward(args, rank, world, local)
    if args.routing == "sigmoid":
        return run_sigmoid(args, rank, world, local)
    return run_native(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
