"""Benchmark of the Permute + GroupedMatMul (+ shared-expert MatMul) hot path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--permute-out] [--path fused|split|default] [--impl reference]

One step = one call of the whole hot path (segment scan, permute, routed
grouped GEMM, shared-expert GEMM) on one rank's synthetic inputs, resident in
HBM.  Prints one JSON line (rank 0).  Metric: algorithmic TFLOP/s,
2 * A * H1 * N1 + 2 * BS * H2 * N2 per step, summed over ranks, divided by the
max over ranks of the device time of the K timed steps.

Under torchrun (N > 1) every rank runs its own expert-parallel rank's share
(its own recvCounts and tensors): weak scaling, no collective on the data path.

--impl reference times the CPU oracle (float64, OpenMP) on the host cores on a
bounded sample of the same workload and prints the same line with
"impl": "reference".

Other measurements (one JSON line each):
    --op amp       the loss-scale step: inf/NaN scan and scale update
    --op qreduce   the dequantising rank reduce [--qworkload NAME]
    --op layer     AlltoAllv (NCCL) + the hot path, per rank [--overlap]
    --op mx        the hot path with block-scaled FP8 operands [--mx-qtype]
    --op arrivals  rows landing source by source while the kernel runs (one GPU)
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from token_permute_grouped_gb300 import binding, build  # noqa: E402
from token_permute_grouped_gb300.workloads import HEADLINE, SMALL, W8E4, WORKLOADS, make_inputs  # noqa: E402

METRIC = "permute+grouped-GEMM TFLOP/s, % of GB300 bf16 dense peak; us per call"
L2_BYTES = 129 * 2**20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


def flops_of(wl, A):
    return 2.0 * A * wl.H1 * wl.N1 + 2.0 * wl.BS * wl.H2 * wl.N2


def algorithmic_bytes(wl, A, permute_out):
    """Each input read once, each output written once (16-bit elements)."""
    b = 2 * (A * wl.H1 + wl.e * wl.H1 * wl.N1 + A * wl.N1)
    b += 2 * (wl.BS * wl.H2 + wl.H2 * wl.N2 + wl.BS * wl.N2)
    b += 4 * wl.W * wl.e
    if permute_out:
        b += 2 * A * wl.H1
    return b


def replicas_for(wl, A, permute_out):
    """Input replicas rotated between steps so that no step finds its inputs in L2."""
    return min(64, max(2, -(-3 * L2_BYTES // max(algorithmic_bytes(wl, A, permute_out), 1))))


def workload_config(wl, A, args):
    """The line's `config`: the workload and the protocol, identical in both arms."""
    reps = replicas_for(wl, A, args.permute_out)
    set_mib = reps * algorithmic_bytes(wl, A, args.permute_out) / 2**20
    return {
        "workload": wl.name, "W": wl.W, "e": wl.e, "A": A, "H1": wl.H1, "N1": wl.N1,
        "BS": wl.BS, "H2": wl.H2, "N2": wl.N2, "dtype": wl.dtype, "path": args.path, "tiles": args.tiles,
        "permute_out": bool(args.permute_out), "accumulate": "fp32",
        "l2": (f"GPU arm: inputs rotated over {reps} replicas ({set_mib:.0f} MiB > 129 MiB L2); "
               "reference arm: host memory"),
    }


# The sources each measured call depends on (kernels and host setup).
GEMM_SOURCES = ("api.cu", "grouped_gemm.cu", "kernels.h", "permute.cu", "plan.cuh", "ptx.cuh")
QREDUCE_SOURCES = ("quant_reduce.cu", "ptx.cuh", "../../include/a2av_quant_reduce.h")
MX_SOURCES = ("grouped_gemm_mx.cu", "plan.cuh", "ptx.cuh", "../../include/a2av_gmm_mx.h")
AMP_SOURCES = ("amp.cu", "kernels.h")


def source_hash(names=GEMM_SOURCES):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "token_permute_grouped_gb300", "csrc", name), "rb") as fh:
            h.update(os.path.basename(name).encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, permute_out=False, path="default", tiles="default", kernel="grouped_gemm_kernel"):
    """DRAM bytes per launch of a kernel from a committed ncu summary, only
    while the kernel's sources are unchanged since the capture."""
    names = {"quant_reduce_kernel": QREDUCE_SOURCES, "grouped_gemm_mx_kernel": MX_SOURCES,
             "nonfinite_scan_kernel": AMP_SOURCES}.get(kernel, GEMM_SOURCES)
    for f in glob.glob(os.path.join(ROOT, "profiles", "*.json")):
        try:
            with open(f) as fh:
                s = json.load(fh)
        except (OSError, ValueError):
            continue
        if (s.get("kernel", "grouped_gemm_kernel") == kernel and s.get("workload") == workload
                and s.get("permute_out", False) == permute_out
                and s.get("path", "default") == path and s.get("tiles", "default") == tiles
                and s.get("source_hash") == source_hash(names)):
            return s.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons, sampled every 20 ms while
    the block runs.  timed_region() marks the timed calls' wall-clock window
    on the active sampler, and summary() reports the samples that fell inside
    those windows (those around them only when none did, and says so)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20
    active = None

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (host time when read, csv line)
        self.windows = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        ClockSampler.active = self
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        ClockSampler.active = None
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def _parse(self, lines):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, pw, mx, reasons = [], [], None, set()
        for _, line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                pw.append(float(parts[3]))
            except ValueError:
                pass
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return sm, pw, mx, reasons

    def summary(self):
        # A line is read a moment after nvidia-smi took the sample: allow one
        # period of slack at the end of each window.
        slack = self.PERIOD_MS / 1e3
        inside = [x for x in self.lines if any(t0 <= x[0] <= t1 + slack for t0, t1 in self.windows)]
        sm, pw, mx, reasons = self._parse(inside)
        basis = "samples taken during the timed calls"
        if not sm:
            sm, pw, mx, reasons = self._parse(self.lines)
            span = sum(t1 - t0 for t0, t1 in self.windows) * 1e3
            basis = f"no sample fell inside the timed calls ({span:.0f} ms): samples around them"
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_total": len(self.lines), "basis": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm), "sm_max_mhz": mx,
                "power_w_median": statistics.median(pw) if pw else None, "reasons": sorted(reasons),
                "samples": len(sm), "samples_total": len(self.lines), "period_ms": self.PERIOD_MS,
                "basis": basis}


# ------------------------------------------------------------ distributed glue

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def timed_region(step, steps, world, device, sync):
    """Barrier + sync on both sides of exactly `steps` calls of step(i);
    returns (this rank's seconds, max over ranks)."""
    barrier(world)
    sync()
    t0 = time.perf_counter()
    w0 = time.time()
    for i in range(steps):
        step(i)
    sync()
    w1 = time.time()
    barrier(world)
    dt = time.perf_counter() - t0
    if ClockSampler.active is not None:
        ClockSampler.active.mark(w0, w1)
    return dt, reduce_max(dt, world, device)


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    world, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a GPU (use --impl reference for the CPU oracle)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    build.build()
    binding.load()

    wl = WORKLOADS[args.workload]
    # One process simulates the expert-parallel rank it stands for: its own
    # rank under torchrun, or --sim-rank on one GPU.
    sim_rank = rank if args.sim_rank is None else args.sim_rank
    inp = make_inputs(wl, seed=0, rank=sim_rank)
    A = inp.A
    dt = wl.torch_dtype
    plan = binding.Plan(wl.W, wl.e, A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt,
                        want_permute_out=args.permute_out, path=args.path, device=dev, tiles=args.tiles)
    launches_per_call = binding.a2av_gmm_launch_count(plan.desc)

    # Input replicas, rotated so that no step finds its inputs in L2.
    reps = replicas_for(wl, A, args.permute_out)
    host = {"ataOut": inp.ataOut, "gmmWeight": inp.gmmWeight, "mmX": inp.mmX, "mmWeight": inp.mmWeight}
    rc_dev = torch.from_numpy(inp.recvCounts).to(dev)
    sets = []
    for _ in range(reps):
        s = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
        s["gmmY"] = torch.empty(A, wl.N1, dtype=dt, device=dev)
        s["mmY"] = torch.empty(wl.BS, wl.N2, dtype=dt, device=dev) if wl.BS else None
        s["perm"] = torch.empty(A, wl.H1, dtype=dt, device=dev) if args.permute_out else None
        sets.append(s)
    stream = torch.cuda.current_stream(dev)

    def step(i, gemm_events=None):
        s = sets[i % reps]
        plan.run(s["ataOut"], rc_dev, s["gmmWeight"], s["mmX"], s["mmWeight"], gmmY=s["gmmY"], mmY=s["mmY"],
                 permuteOut=s["perm"], stream=stream, gemm_events=gemm_events)

    sync = torch.cuda.synchronize
    for i in range(args.warmup):
        step(i)
    sync()
    st, code = binding.a2av_gmm_read_device_status(plan.workspace)
    if st != 0:
        raise RuntimeError(f"device status {st} ({code})")

    # Per-call device time on the launching stream: the whole call (scan,
    # permute and GEMM), which `value` reports.
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]

    def timed_step(i):
        if i == 0:
            ev[0].record(stream)
        step(i)
        ev[i + 1].record(stream)

    with ClockSampler(local) as clocks:
        wall, wall_max = timed_region(timed_step, args.steps, world, dev, sync)
    per_call_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    dev_s = sum(per_call_ms) / 1e3
    dev_s_max = reduce_max(dev_s, world, dev)
    flops = flops_of(wl, A)
    total_flops = reduce_sum(flops * args.steps, world, dev)
    tflops = total_flops / dev_s_max / 1e12
    ms_per_step = dev_s_max * 1e3 / args.steps

    # The dominant kernel alone: K more calls through a2av_gmm_run_profiled,
    # which records a pair of events on the launching stream right around the
    # grouped-GEMM kernel (the GEMM then starts after the permute kernel in
    # plain stream order).
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    timed_region(lambda i: step(i, gev[i]), args.steps, world, dev, sync)
    gemm_ms = [b.elapsed_time(e) for b, e in gev]

    # End to end through the same public call with host buffers: this step's
    # activations (ataOut, recvCounts, mmX) copied in from pinned memory, the
    # results (gmmY, mmY) read back.  Weights stay resident, as in a model.
    pin = {k: (v.pin_memory() if v is not None else None) for k, v in
           {"ataOut": inp.ataOut, "mmX": inp.mmX}.items()}
    rc_pin = torch.from_numpy(inp.recvCounts).pin_memory()
    out_y = torch.empty(A, wl.N1, dtype=dt).pin_memory()
    out_mm = torch.empty(wl.BS, wl.N2, dtype=dt).pin_memory() if wl.BS else None
    h2d = pin["ataOut"].numel() * 2 + rc_pin.numel() * 4 + (pin["mmX"].numel() * 2 if wl.BS else 0)
    d2h = out_y.numel() * 2 + (out_mm.numel() * 2 if wl.BS else 0)

    # Two device buffer sets: step i+1's inputs are copied in on their own
    # stream while step i computes; step i's results go out on a third.
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    bufs = [sets[0], sets[1 % reps]]
    rcs = [rc_dev, torch.empty_like(rc_dev)]
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def issue_h2d(b):
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(comp_done[b])  # the previous user of set b has read it
            bufs[b]["ataOut"].copy_(pin["ataOut"], non_blocking=True)
            rcs[b].copy_(rc_pin, non_blocking=True)
            if wl.BS:
                bufs[b]["mmX"].copy_(pin["mmX"], non_blocking=True)
            h2d_done[b].record(h2d_stream)

    def e2e_step(i):
        b = i % 2
        if i == 0:
            issue_h2d(0)
        stream.wait_event(h2d_done[b])
        stream.wait_event(d2h_done[b])  # set b's outputs from step i-2 are out
        s = bufs[b]
        plan.run(s["ataOut"], rcs[b], s["gmmWeight"], s["mmX"], s["mmWeight"], gmmY=s["gmmY"], mmY=s["mmY"],
                 permuteOut=s["perm"], stream=stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(comp_done[b])
            out_y.copy_(s["gmmY"], non_blocking=True)
            if wl.BS:
                out_mm.copy_(s["mmY"], non_blocking=True)
            d2h_done[b].record(d2h_stream)
        if i + 1 < e2e_steps:
            issue_h2d(1 - b)

    e2e_steps = 1
    e2e_step(0)
    sync()
    e2e_steps = max(3, min(args.steps, 20))
    _, e2e_max = timed_region(e2e_step, e2e_steps, world, dev, sync)
    e2e_tflops = reduce_sum(flops * e2e_steps, world, dev) / e2e_max / 1e12

    # Sustained: the same call back to back for about --sustained-s seconds
    # (power draw settles and the 1.4 kW cap may lower the SM clock), timed
    # as a whole with two events; reported beside the burst figures above.
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, int(args.sustained_s * 1e3 / max(ms_per_step, 1e-3)))
        sus_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

        def sus_step(i):
            if i == 0:
                sus_ev[0].record(stream)
            step(i)
            if i == n_sus - 1:
                sus_ev[1].record(stream)

        with ClockSampler(local) as sus_clocks:
            timed_region(sus_step, n_sus, world, dev, sync)
        sus_s = reduce_max(sus_ev[0].elapsed_time(sus_ev[1]) / 1e3, world, dev)
        sustained = {"calls": n_sus, "us_per_call": round(sus_s * 1e6 / n_sus, 2),
                     "tflops": round(reduce_sum(flops * n_sus, world, dev) / sus_s / 1e12, 2),
                     "clocks": sus_clocks.summary()}

    if rank != 0:
        barrier(world)
        return
    pk, pk_kind = peaks()
    peak_tf = pk["bf16_tflops"]
    gemm_s = statistics.fmean(gemm_ms) / 1e3
    achieved = flops / gemm_s / 1e12
    whole = flops / (dev_s / args.steps) / 1e12
    line = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded routing and N(0,1) tensors; no dataset)",
        "config": {**workload_config(wl, A, args), **({"sim_rank": sim_rank} if args.sim_rank is not None else {})},
        "timing": {
            "us_per_call_median": round(statistics.median(per_call_ms) * 1e3, 2),
            "us_per_call_min": round(min(per_call_ms) * 1e3, 2),
            "us_per_call_p90": round(float(np.percentile(per_call_ms, 90)) * 1e3, 2),
            "gemm_kernel_us_mean": round(gemm_s * 1e6, 2),
            "gemm_kernel_us_p90": round(float(np.percentile(gemm_ms, 90)) * 1e3, 2),
            "pct_of_bf16_peak": round(100 * tflops / world / peak_tf, 2),
            "pct_of_bf16_sustained": round(100 * tflops / world / pk["bf16_tflops_sustained"], 2),
            "gflop_per_call": round(flops / 1e9, 3),
            "group_rows": inp.recvCounts.reshape(wl.W, wl.e).sum(0).tolist(),
            "launches_per_call": launches_per_call,
        },
        "roofline": {
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "peak": peak_tf,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak_tf, 4),
            "traffic": profiled_traffic(wl.name, bool(args.permute_out), args.path, args.tiles),
            "kernel": "grouped_gemm_kernel",
            "timed": ("the GEMM kernel alone: CUDA events recorded on its launching stream right before and "
                      f"after it, mean of {args.steps} launches (a2av_gmm_run_profiled)"),
            "whole_call": {"achieved": round(whole, 2), "frac": round(whole / peak_tf, 4),
                           "timed": "scan + permute + GEMM, CUDA events around each call"},
            "peak_source": f"{pk_kind} bf16 dense burst (MEASURED_PEAKS.json bf16_tflops)" if pk_kind == "measured"
            else "fallback 1.9 PFLOP/s",
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes": algorithmic_bytes(wl, A, args.permute_out),
        },
        "e2e": {"value": round(e2e_tflops, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "inputs_copied": "ataOut, recvCounts, mmX from pinned host memory (weights resident)",
                "overlap": "step i+1's H2D and step i's D2H run on copy streams beside step i's kernels"},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": clocks.summary(),
    }
    if sustained is not None:
        sustained["frac_of_bf16_sustained"] = round(sustained["tflops"] / world / pk["bf16_tflops_sustained"], 4)
        sustained["timed"] = ("the same call back to back, outside the K timed steps; CUDA events around the "
                              "whole run; peak: MEASURED_PEAKS.json bf16_tflops_sustained")
        line["sustained"] = sustained
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_seconds)
    emit(line)
    barrier(world)


# --------------------------------------------------------------- CPU oracle

def oracle_sample(wl, inp, seconds, seed=0):
    """Time the oracle on a seeded sample of output rows; returns
    (FLOPs done, seconds, rows, threads, description).  The oracle's permute
    (a copy of every row) runs once, untimed, to give it its own input."""
    import oracle
    orc = oracle.Oracle()
    A = inp.A
    perm = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut)
    _, _, gr, _ = orc.plan(wl.W, wl.e, inp.recvCounts, A)
    rng = np.random.default_rng(seed)
    per_row_routed = 2.0 * wl.H1 * wl.N1
    per_row_shared = 2.0 * wl.H2 * wl.N2
    total_rows = A + wl.BS
    chunk = max(orc.num_threads(), 8)
    flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds and rows_done < total_rows:
        r = rng.integers(0, total_rows, chunk)
        routed = r[r < A]
        shared = r[r >= A] - A
        if len(routed):
            orc.grouped_matmul(gr, perm, inp.gmmWeight, routed)
            flops += per_row_routed * len(routed)
        if len(shared):
            orc.matmul(inp.mmX, inp.mmWeight, shared)
            flops += per_row_shared * len(shared)
        rows_done += chunk
    el = time.perf_counter() - t0
    desc = (f"{rows_done} output rows drawn uniformly from the {total_rows} rows of gmmY and mmY "
            f"of {wl.name} (float64 oracle, full K per row)")
    return flops, el, rows_done, orc.num_threads(), desc


def cpu_baseline(wl, inp, seconds):
    flops, el, rows, threads, desc = oracle_sample(wl, inp, seconds)
    line = {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": desc, "seconds": round(el, 2)}
    if wl.name in (SMALL, W8E4):
        # The same oracle on one core, beside all of them.
        import oracle
        orc = oracle.Oracle()
        all_threads = orc.num_threads()
        orc.set_threads(1)
        try:
            f1, el1, _, _, desc1 = oracle_sample(wl, inp, seconds / 3, seed=1)
        finally:
            orc.set_threads(all_threads)
        line["one_thread"] = {"value": round(f1 / el1 / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "sample": desc1,
                              "seconds": round(el1, 2)}
    return line


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # rank 0 alone times the oracle
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl, seed=0)
    per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, inp, per_step / 4)
    tot_f = tot_s = 0.0
    threads = 1
    desc = ""
    for i in range(args.steps):
        f, s, _, threads, desc = oracle_sample(wl, inp, per_step, seed=i + 1)
        tot_f += f
        tot_s += s
    tf = tot_f / tot_s / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(tf, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, inp.A, args),
        "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc, "seconds_per_step": per_step},
        "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    emit(line)


def run_amp(args):
    """Loss-scale step: the inf/NaN scan over a layer output (HBM-bound) and
    the scalar update ("aclnnAmpUpdateScale"), timed with CUDA events."""
    assert torch.cuda.is_available()
    dev = torch.device("cuda", 0)
    build.build()
    binding.load()
    n = 34502 * 4096  # the DeepSeek-V3-like gmmY: 283 MB of bf16
    bufs = [torch.randn(n, device=dev, dtype=torch.float32).to(torch.bfloat16) for _ in range(2)]
    flag = torch.zeros(1, device=dev)
    scale = torch.tensor([65536.0], device=dev)
    tracker = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        binding.a2av_found_nonfinite(bufs[i % 2], flag)
        binding.a2av_amp_update_scale(scale, tracker, flag, 2.0, 0.5, 2000)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with ClockSampler(0) as clocks:
        ev[0].record(stream)
        for i in range(args.steps):
            binding.a2av_found_nonfinite(bufs[i % 2], flag)
        ev[1].record(stream)
        for i in range(args.steps):
            binding.a2av_amp_update_scale(scale, tracker, flag, 2.0, 0.5, 2000)
        ev[2].record(stream)
        torch.cuda.synchronize()
    scan_s = ev[0].elapsed_time(ev[1]) / 1e3 / args.steps
    upd_us = ev[1].elapsed_time(ev[2]) * 1e3 / args.steps
    gbs = n * 2 / scan_s / 1e9
    pk, pk_kind = peaks()
    emit({
        "metric": "loss-scale step: inf/NaN scan GB/s over a bf16 layer output; us per scale update",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(scan_s * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic N(0,1)",
        "config": {"workload": "amp_scan_bf16_34502x4096", "bytes_per_scan": n * 2,
                   "l2": "two 283 MB buffers alternated (> 129 MiB L2)", "update_us_per_call": round(upd_us, 2)},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / pk["hbm_gbs"], 4),
                     "traffic": profiled_traffic("amp_scan_bf16_34502x4096", kernel="nonfinite_scan_kernel"),
                     "kernel": "nonfinite_scan_kernel",
                     "peak_source": f"{pk_kind} copy bandwidth (read + write); the scan only reads"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
    })


# ----------------------------------------------------------- quantised reduce

QR_METRIC = "quantised rank reduce: algorithmic GB/s (8-bit codes + scales in, bf16 out)"


def qreduce_bytes(wl):
    """Algorithmic bytes of one call: every code and scale read once, the output written once."""
    n = wl.W * wl.rows * wl.H
    scale_bytes = n // 32 if wl.mode == "mx" else n // 128 * 4
    return n + scale_bytes + wl.rows * wl.H * 2


def qreduce_oracle_sample(wl, data, scales, seconds, seed=0):
    """Oracle on seeded batches of output rows (rows reduce independently); returns
    (algorithmic bytes covered, seconds, rows, threads, description)."""
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(seed)
    qt = {"e4m3fn": 0, "e5m2": 1, "int8": 2}[wl.qtype]
    mode = 0 if wl.mode == "mx" else 1
    per_row = qreduce_bytes(wl) / wl.rows
    chunk = max(orc.num_threads(), 8)
    rows = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        idx = rng.integers(0, wl.rows, chunk)
        orc.quant_reduce(np.ascontiguousarray(data[:, idx]), np.ascontiguousarray(scales[:, idx]), qt, mode)
        rows += chunk
    el = time.perf_counter() - t0
    desc = (f"{rows} output rows drawn uniformly, with repeats, from the {wl.rows} rows of {wl.name} "
            f"(float64 oracle)")
    return per_row * rows, el, rows, orc.num_threads(), desc


def run_qreduce(args):
    """Dequantising rank reduce ("aclnnQuantReduceScatter" page), one launch per step, HBM-bound.
    Under torchrun every rank reduces its own received data: weak scaling, no collective."""
    from token_permute_grouped_gb300.workloads import QREDUCE_WORKLOADS, quant_reduce_inputs
    world, rank, local = dist_env()
    wl = QREDUCE_WORKLOADS[args.qworkload]
    if args.impl == "reference":
        if rank != 0:
            return
        data, scales = (t.numpy() for t in quant_reduce_inputs(wl.W, wl.rows, wl.H, wl.qtype, wl.mode, seed=0))
        per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
        for _ in range(args.warmup):
            qreduce_oracle_sample(wl, data, scales, per_step / 4)
        tot_b = tot_s = 0.0
        threads, desc = 1, ""
        for i in range(args.steps):
            b, sec, _, threads, desc = qreduce_oracle_sample(wl, data, scales, per_step, seed=i + 1)
            tot_b += b
            tot_s += sec
        gbs = tot_b / tot_s / 1e9
        emit({
            "impl": "reference", "metric": QR_METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s * 1e3 / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "W": wl.W, "rows": wl.rows, "H": wl.H, "qtype": wl.qtype,
                       "mode": wl.mode, "seconds_per_step": per_step},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        })
        return
    assert torch.cuda.is_available(), "bench.py needs a GPU (use --impl reference for the CPU oracle)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    build.build()
    binding.load()
    data, scales = quant_reduce_inputs(wl.W, wl.rows, wl.H, wl.qtype, wl.mode, seed=rank)
    nbytes = qreduce_bytes(wl)
    reps = min(64, max(2, -(-3 * L2_BYTES // nbytes)))
    sets = [(data.to(dev), scales.to(dev), torch.empty(wl.rows, wl.H, dtype=torch.bfloat16, device=dev))
            for _ in range(reps)]
    stream = torch.cuda.current_stream(dev)

    def step(i):  # on the current stream (the graph's capture stream while capturing)
        d, sc, o = sets[i % reps]
        binding.a2av_quant_reduce(d, sc, wl.qtype, wl.mode, o)

    sync = torch.cuda.synchronize
    for i in range(args.warmup):
        step(i)
    sync()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    # Eager: the K calls launched one by one from Python.  A call's kernel
    # takes about as long as its host-side argument checks and launch, so
    # this also measures the launch path.
    def timed_step(i):
        if i == 0:
            ev[0].record(stream)
        step(i)
        if i == args.steps - 1:
            ev[1].record(stream)

    timed_region(timed_step, args.steps, world, dev, sync)
    eager_s = ev[0].elapsed_time(ev[1]) / 1e3
    # The same K calls captured in one CUDA graph and replayed: device time
    # of the kernels back to back, which the value reports.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            step(i)
    graph.replay()
    sync()

    def replay(_):
        ev[0].record(stream)
        graph.replay()
        ev[1].record(stream)

    with ClockSampler(local) as clocks:
        timed_region(replay, 1, world, dev, sync)
    dev_s = ev[0].elapsed_time(ev[1]) / 1e3
    dev_s_max = reduce_max(dev_s, world, dev)
    gbs = reduce_sum(nbytes * args.steps, world, dev) / dev_s_max / 1e9

    # End to end through the same call with host buffers: codes and scales in
    # from pinned memory, the reduced rows back out, on copy streams that
    # overlap the neighbouring steps' kernels (two device buffer sets).
    pin_d, pin_s = data.pin_memory(), scales.pin_memory()
    out_h = torch.empty(wl.rows, wl.H, dtype=torch.bfloat16).pin_memory()
    h2d_b = pin_d.numel() + pin_s.numel() * pin_s.element_size()
    d2h_b = out_h.numel() * 2
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))

    def issue_h2d(b):
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(comp_done[b])
            sets[b][0].copy_(pin_d, non_blocking=True)
            sets[b][1].copy_(pin_s, non_blocking=True)
            h2d_done[b].record(h2d_stream)

    def e2e_step(i):
        b = i % 2
        if i == 0:
            issue_h2d(0)
        stream.wait_event(h2d_done[b])
        stream.wait_event(d2h_done[b])
        d, sc, o = sets[b]
        binding.a2av_quant_reduce(d, sc, wl.qtype, wl.mode, o, stream=stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(comp_done[b])
            out_h.copy_(o, non_blocking=True)
            d2h_done[b].record(d2h_stream)
        if i + 1 < e2e_steps:
            issue_h2d(1 - b)

    _, e2e_max = timed_region(e2e_step, e2e_steps, world, dev, sync)
    e2e_gbs = reduce_sum(nbytes * e2e_steps, world, dev) / e2e_max / 1e9
    if rank != 0:
        barrier(world)
        return
    pk, pk_kind = peaks()
    achieved = nbytes / (dev_s / args.steps) / 1e9
    line = {
        "metric": QR_METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dev_s_max * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded uniform finite codes, power-of-two or 2^u scales; no dataset)",
        "config": {"workload": wl.name, "W": wl.W, "rows": wl.rows, "H": wl.H, "qtype": wl.qtype, "mode": wl.mode,
                   "out": "bf16", "accumulate": "fp32", "bytes_per_call": nbytes,
                   "us_per_call": round(dev_s / args.steps * 1e6, 2),
                   "timing": "the K calls captured in one CUDA graph and replayed (CUDA events around the replay)",
                   "eager_us_per_call": round(eager_s / args.steps * 1e6, 2),
                   "l2": (f"inputs rotated over {reps} replicas ({reps * nbytes / 2**20:.0f} MiB > 129 MiB L2)"
                          if reps * nbytes > L2_BYTES else
                          f"all {reps} replicas ({reps * nbytes / 2**20:.0f} MiB) fit in L2: a latency-bound case")},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4),
                     "traffic": profiled_traffic(wl.name, kernel="quant_reduce_kernel"),
                     "kernel": "quant_reduce_kernel",
                     "peak_source": f"{pk_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if pk_kind == "measured"
                     else "fallback 6.8 TB/s", "algorithmic_bytes": nbytes},
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d_b),
                "d2h_bytes_per_step": int(d2h_b), "steps": e2e_steps,
                "inputs_copied": "codes and scales from pinned host memory; output read back"},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        b, sec, _, threads, desc = qreduce_oracle_sample(wl, data.numpy(), scales.numpy(), args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(b / sec / 1e9, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": desc, "seconds": round(sec, 2)}
    emit(line)
    barrier(world)


# ------------------------------------------------------ the whole operator

def run_layer(args):
    """AlltoAllv (NCCL) + Permute + GroupedMatMul + shared-expert MatMul per step, through
    exchange.layer.  Every rank sends its gmmX rows to their expert owners, so with N ranks
    this is the full expert-parallel exchange (N = 1: rows go to the same rank)."""
    from token_permute_grouped_gb300 import exchange
    from token_permute_grouped_gb300.workloads import Workload, make_gmmX
    world, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a GPU (use --impl reference for the CPU oracle)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not torch.distributed.is_initialized():
        if world == 1:
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", str(29500 + os.getpid() % 1000))
            torch.distributed.init_process_group("nccl", rank=0, world_size=1)
        else:
            torch.distributed.init_process_group("nccl")
    build.build()
    binding.load()
    base = WORKLOADS[args.workload]
    if base.routing != "normal":
        raise SystemExit(f"--op layer needs a workload with the normal routing model, not {base.name}")
    # The expert-parallel domain is the torchrun world: W = N ranks with the workload's e, H, N.
    # With fewer than K global experts, K is capped at W*e and each source routes
    # proportionally more tokens, so a rank still expects tokens_per_source * K rows.
    k = min(base.topk, world * base.e)
    wl = Workload(f"{base.name}_ep{world}", W=world, e=base.e, H1=base.H1, N1=base.N1, dtype=base.dtype,
                  routing="normal", tokens_per_source=base.tokens_per_source * base.topk // k, topk=k,
                  bias_std=base.bias_std, BS=base.BS, H2=base.H2, N2=base.N2)
    gmmX, sc = make_gmmX(wl, seed=0, rank=rank)
    inp = make_inputs(base, seed=0, rank=rank)  # weights and mmX of this rank
    reps = 2
    sets = [dict(gmmX=gmmX.to(dev), sc=torch.from_numpy(sc).to(dev), gw=inp.gmmWeight.to(dev),
                 mmX=inp.mmX.to(dev) if wl.BS else None, mmW=inp.mmWeight.to(dev) if wl.BS else None)
            for _ in range(reps)]
    out = {}

    def step(i):
        s = sets[i % reps]
        out["r"] = exchange.layer(s["gmmX"], s["sc"], s["gw"], s["mmX"], s["mmW"],
                                  overlap_shared=args.overlap)

    sync = torch.cuda.synchronize
    for i in range(args.warmup):
        step(i)
    sync()
    A = int(out["r"][3].shape[0])
    flops = flops_of(wl, A)
    with ClockSampler(local) as clocks:
        dt, dt_max = timed_region(step, args.steps, world, dev, sync)
    total = reduce_sum(flops * args.steps, world, dev)
    tflops = total / dt_max / 1e12
    plan = binding.Plan(wl.W, wl.e, A, wl.H1, wl.N1, 0 if args.overlap else wl.BS, wl.H2, wl.N2,
                        wl.torch_dtype, device=dev)
    launches = binding.a2av_gmm_launch_count(plan.desc) + (1 if wl.BS and args.overlap else 0)
    if rank != 0:
        barrier(world)
        return
    pk, pk_kind = peaks()
    emit({
        "metric": METRIC + " (with the AlltoAllv in the step)", "value": round(tflops, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt_max * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded routing and N(0,1) tensors; no dataset)",
        "config": {"workload": wl.name, "W": wl.W, "e": wl.e, "A_rank0": A, "H1": wl.H1, "N1": wl.N1,
                   "tokens_per_source": wl.tokens_per_source, "topk": wl.topk,
                   "BS": wl.BS, "H2": wl.H2, "N2": wl.N2,
                   "exchange": f"NCCL all_to_all_single of counts, then of rows, world {world}",
                   "shared_expert": "beside the row exchange" if args.overlap else "with the routed experts",
                   "timing": "host wall clock between barriers and syncs (the step syncs once on the counts)",
                   "l2": f"inputs rotated over {reps} replicas (gmmX alone {gmmX.numel() * 2 / 2**20:.0f} MiB)"},
        "roofline": {"bound": "tensor", "achieved": round(tflops / world, 2), "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(tflops / world / pk["bf16_tflops"], 4), "traffic": None,
                     "peak_source": f"{pk_kind} bf16 dense burst", "note": "per GPU, exchange included"},
        "e2e": None,
        "gpu_launches": launches * args.steps,
        "clocks": clocks.summary(),
    })
    barrier(world)


# ------------------------------------- arrival-driven start (emulated exchange)

ARR_METRIC = ("AlltoAllv landing + permute+grouped-GEMM TFLOP/s per step, rows arriving while the kernel runs "
              "(exchange emulated by host-to-device copies); us per step")


def run_arrivals(args):
    """One GPU: each step's received rows land in ataOut source by source (copies from pinned host
    memory on a side stream, each followed by its source's flag) while a2av_gmm_run_arrivals runs on
    the compute stream; beside it, the same step in sequence (all rows copied, then the default call)."""
    world, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    binding.load()
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl, seed=0, rank=rank)
    A, dt = inp.A, wl.torch_dtype
    per_source = inp.recvCounts.reshape(wl.W, wl.e).astype(np.int64).sum(1)
    ends = np.cumsum(per_source)
    spans = [(int(b), int(t)) for b, t in zip(ends - per_source, ends)]
    host = inp.ataOut.pin_memory()
    ata = torch.empty(A, wl.H1, dtype=dt, device=dev)
    rc = torch.from_numpy(inp.recvCounts).to(dev)
    gw = inp.gmmWeight.to(dev)
    mmX = inp.mmX.to(dev) if wl.BS else None
    mmW = inp.mmWeight.to(dev) if wl.BS else None
    y = torch.empty(A, wl.N1, dtype=dt, device=dev)
    my = torch.empty(wl.BS, wl.N2, dtype=dt, device=dev) if wl.BS else None
    arrived = torch.zeros(wl.W, dtype=torch.int64, device=dev)
    n_all = args.warmup + args.steps
    tags = torch.arange(1, 2 * n_all + 1, dtype=torch.int64).mul_(0x9E3779B9).pin_memory()
    desc = binding.make_desc(wl.W, wl.e, A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt, path="fused")
    ws = torch.empty(binding.a2av_gmm_workspace_size(desc), dtype=torch.uint8, device=dev)
    plan = binding.Plan(wl.W, wl.e, A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, dt, device=dev)
    main = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    done = [torch.cuda.Event() for _ in range(2)]
    landed = torch.cuda.Event()

    def land(i, flags):
        # the exchange's rows for step i, source by source; each source's flag after its rows
        with torch.cuda.stream(side):
            side.wait_event(done[(i - 1) % 2])  # the previous step has read ataOut
            for w, (b, t) in enumerate(spans):
                if t > b:
                    ata[b:t].copy_(host[b:t], non_blocking=True)
                if flags:
                    arrived[w:w + 1].copy_(tags[i:i + 1], non_blocking=True)
            landed.record(side)

    def overlapped(i):
        land(i, True)
        binding.a2av_gmm_run_arrivals(desc, ata, rc, gw, mmX, mmW, None, y, my, arrived, int(tags[i]), 0, ws,
                                      stream=main)
        done[i % 2].record(main)

    def sequential(i):
        land(i, False)
        main.wait_event(landed)
        plan.run(ata, rc, gw, mmX, mmW, gmmY=y, mmY=my, stream=main)
        done[i % 2].record(main)

    sync = torch.cuda.synchronize
    for i in range(2):
        done[i].record(main)
    res = {}
    for name, fn, base in (("overlapped", overlapped, 0), ("sequential", sequential, n_all)):
        for i in range(args.warmup):
            fn(base + i)
        sync()
        with ClockSampler(local) as clocks:
            dt_s, _ = timed_region(lambda i: fn(base + args.warmup + i), args.steps, world, dev, sync)
        res[name] = (dt_s, clocks.summary())
    st, code = binding.a2av_gmm_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} ({code})")
    flops = flops_of(wl, A)
    h2d = sum(t - b for b, t in spans) * wl.H1 * 2 + wl.W * 8
    ov, sq = res["overlapped"][0] / args.steps, res["sequential"][0] / args.steps
    pk, pk_kind = peaks()
    emit({
        "metric": ARR_METRIC, "value": round(flops / ov / 1e12, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ov * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded routing and N(0,1) tensors; no dataset)",
        "config": {"workload": wl.name, "W": wl.W, "e": wl.e, "A": A, "H1": wl.H1, "N1": wl.N1, "BS": wl.BS,
                   "H2": wl.H2, "N2": wl.N2, "dtype": wl.dtype,
                   "exchange": "rows of each source copied host-to-device from pinned memory on a side stream, "
                               "then that source's 8-byte flag",
                   "l2": "ataOut rewritten by the copies every step"},
        "timing": {"us_per_step_overlapped": round(ov * 1e6, 2), "us_per_step_sequential": round(sq * 1e6, 2),
                   "sequential": "all rows copied, then the default call (split_runs)",
                   "overlapped": "a2av_gmm_run_arrivals (fused path) launched beside the copies",
                   "h2d_bytes_per_step": int(h2d), "h2d_gbs_overlapped": round(h2d / ov / 1e9, 1)},
        "roofline": {"bound": "hbm", "achieved": round(h2d / ov / 1e9, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": None, "traffic": None,
                     "note": "bound by the host-to-device link, not by HBM or the tensor cores"},
        "e2e": {"value": round(flops / ov / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": 0},
        "gpu_launches": args.steps,
        "clocks": res["overlapped"][1],
    })


# ------------------------------------------------ block-scaled FP8 (mx) GEMM

MX_METRIC = "mx (block-scaled FP8) permute+grouped-GEMM TFLOP/s, % of GB300 FP8 dense peak; us per call"


def mx_bytes(wl, A):
    """Algorithmic bytes of one mx call: codes and E8M0 scales read once (1 + 1/32 bytes per
    element), bf16 outputs written once, permuteOut not requested."""
    ins = A * wl.H1 + wl.e * wl.H1 * wl.N1 + (wl.BS * wl.H2 + wl.H2 * wl.N2 if wl.BS else 0)
    return int(ins * (1 + 1 / 32) + 2 * (A * wl.N1 + wl.BS * wl.N2))


def mx_oracle_sample(wl, inp, seconds, seed=0):
    """Oracle on seeded output rows of the mx call; returns (FLOPs, seconds, rows, threads, description)."""
    import oracle
    orc = oracle.Oracle()
    q = 0 if inp.qtype == "e4m3fn" else 1
    pq = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut_q.view(torch.int16)).view(torch.uint8)
    ps = orc.permute(wl.W, wl.e, inp.recvCounts, inp.ataOut_s.view(torch.int16)).view(torch.uint8)
    _, _, gr, _ = orc.plan(wl.W, wl.e, inp.recvCounts, inp.A)
    rng = np.random.default_rng(seed)
    total_rows = inp.A + wl.BS
    chunk = max(orc.num_threads(), 8)
    flops = 0.0
    rows = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        r = rng.integers(0, total_rows, chunk)
        routed, shared = r[r < inp.A], r[r >= inp.A] - inp.A
        if len(routed):
            orc.mx_grouped_matmul(gr, pq, ps, inp.gmmWeight_q, inp.gmmWeight_s, q, q, routed)
            flops += 2.0 * wl.H1 * wl.N1 * len(routed)
        if len(shared):
            orc.mx_grouped_matmul([wl.BS], inp.mmX_q, inp.mmX_s, inp.mmWeight_q[None], inp.mmWeight_s[None], q, q,
                                  shared)
            flops += 2.0 * wl.H2 * wl.N2 * len(shared)
        rows += chunk
    el = time.perf_counter() - t0
    desc = (f"{rows} output rows drawn uniformly, with repeats, from the {total_rows} rows of gmmY and mmY of "
            f"{wl.name} in mx {inp.qtype} (float64 oracle, full K per row)")
    return flops, el, rows, orc.num_threads(), desc


def run_mx(args):
    """The hot path with block-scaled FP8 operands (a2av_gmm_mx_run), weak scaling under torchrun."""
    from token_permute_grouped_gb300.workloads import make_mx_inputs
    world, rank, local = dist_env()
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        if rank != 0:
            return
        inp = make_mx_inputs(wl, seed=0, qtype=args.mx_qtype)
        per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
        for _ in range(args.warmup):
            mx_oracle_sample(wl, inp, per_step / 4)
        tot_f = tot_s = 0.0
        threads, desc = 1, ""
        for i in range(args.steps):
            f, sec, _, threads, desc = mx_oracle_sample(wl, inp, per_step, seed=i + 1)
            tot_f += f
            tot_s += sec
        tf = tot_f / tot_s / 1e12
        emit({
            "impl": "reference", "metric": MX_METRIC, "value": round(tf, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s * 1e3 / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name + "_mx_" + args.mx_qtype, "A": inp.A, "seconds_per_step": per_step},
            "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0})
        return
    assert torch.cuda.is_available(), "bench.py needs a GPU (use --impl reference for the CPU oracle)"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    build.build()
    binding.load()
    inp = make_mx_inputs(wl, seed=0, rank=rank, qtype=args.mx_qtype)
    A = inp.A
    mx_tiles = args.tiles if args.tiles in ("default", "single", "pair") else "default"
    plan = binding.MxPlan(wl.W, wl.e, A, wl.H1, wl.N1, wl.BS, wl.H2, wl.N2, args.mx_qtype, device=dev, tiles=mx_tiles)
    nbytes = mx_bytes(wl, A)
    reps = min(64, max(2, -(-3 * L2_BYTES // nbytes)))
    names = ("ataOut_q", "ataOut_s", "gmmWeight_q", "gmmWeight_s", "mmX_q", "mmX_s", "mmWeight_q", "mmWeight_s")
    sets = []
    for _ in range(reps):
        st = {k: (getattr(inp, k).to(dev) if getattr(inp, k) is not None else None) for k in names}
        st["gmmY"] = torch.empty(A, wl.N1, dtype=torch.bfloat16, device=dev)
        st["mmY"] = torch.empty(wl.BS, wl.N2, dtype=torch.bfloat16, device=dev) if wl.BS else None
        sets.append(st)
    rc_dev = torch.from_numpy(inp.recvCounts).to(dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, gemm_events=None):
        st = sets[i % reps]
        plan.run(st["ataOut_q"], st["ataOut_s"], rc_dev, st["gmmWeight_q"], st["gmmWeight_s"], st["mmX_q"],
                 st["mmX_s"], st["mmWeight_q"], st["mmWeight_s"], gmmY=st["gmmY"], mmY=st["mmY"], stream=stream,
                 gemm_events=gemm_events)

    sync = torch.cuda.synchronize
    for i in range(args.warmup):
        step(i)
    sync()
    code = binding.a2av_gmm_read_device_status(plan.workspace)
    if code[0] != 0:
        raise RuntimeError(f"device status {code}")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]

    def timed_step(i):
        if i == 0:
            ev[0].record(stream)
        step(i)
        ev[i + 1].record(stream)

    with ClockSampler(local) as clocks:
        timed_region(timed_step, args.steps, world, dev, sync)
    per_call_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    dev_s = sum(per_call_ms) / 1e3
    dev_s_max = reduce_max(dev_s, world, dev)
    flops = flops_of(wl, A)
    tflops = reduce_sum(flops * args.steps, world, dev) / dev_s_max / 1e12

    # The dominant kernel alone, as in the bf16 line: K more calls through
    # a2av_gmm_mx_run_profiled, whose events sit right around the GEMM.
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    timed_region(lambda i: step(i, gev[i]), args.steps, world, dev, sync)
    gemm_ms = [b.elapsed_time(e) for b, e in gev]

    # End to end through the same call: codes and scales of this step's
    # activations (and recvCounts, mmX) in from pinned memory, the bf16
    # results back out; weights resident.  As in the bf16 line, step i + 1's
    # copies in and step i's copies out run on copy streams beside step i's
    # kernels, over two device buffer sets.
    pin = {k: getattr(inp, k).pin_memory() for k in ("ataOut_q", "ataOut_s", "mmX_q", "mmX_s")
           if getattr(inp, k) is not None}
    rc_pin = torch.from_numpy(inp.recvCounts).pin_memory()
    out_y = torch.empty(A, wl.N1, dtype=torch.bfloat16).pin_memory()
    out_m = torch.empty(wl.BS, wl.N2, dtype=torch.bfloat16).pin_memory() if wl.BS else None
    h2d = sum(t.numel() for t in pin.values()) + rc_pin.numel() * 4
    d2h = out_y.numel() * 2 + (out_m.numel() * 2 if wl.BS else 0)
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [sets[0], sets[1 % reps]]
    rcs = [rc_dev, torch.empty_like(rc_dev)]
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))

    def issue_h2d(b):
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(comp_done[b])
            for k, t in pin.items():
                bufs[b][k].copy_(t, non_blocking=True)
            rcs[b].copy_(rc_pin, non_blocking=True)
            h2d_done[b].record(h2d_stream)

    def e2e_step(i):
        b = i % 2
        if i == 0:
            issue_h2d(0)
        stream.wait_event(h2d_done[b])
        stream.wait_event(d2h_done[b])
        st = bufs[b]
        plan.run(st["ataOut_q"], st["ataOut_s"], rcs[b], st["gmmWeight_q"], st["gmmWeight_s"], st["mmX_q"],
                 st["mmX_s"], st["mmWeight_q"], st["mmWeight_s"], gmmY=st["gmmY"], mmY=st["mmY"], stream=stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(comp_done[b])
            out_y.copy_(st["gmmY"], non_blocking=True)
            if wl.BS:
                out_m.copy_(st["mmY"], non_blocking=True)
            d2h_done[b].record(d2h_stream)
        if i + 1 < e2e_steps:
            issue_h2d(1 - b)

    _, e2e_max = timed_region(e2e_step, e2e_steps, world, dev, sync)
    e2e_tflops = reduce_sum(flops * e2e_steps, world, dev) / e2e_max / 1e12
    if rank != 0:
        barrier(world)
        return
    pk, pk_kind = peaks()
    peak = 2.0 * pk["bf16_tflops"]  # FP8 dense = 2x bf16 dense (nominal 4.5 vs 2.25 PFLOP/s)
    gemm_s = statistics.fmean(gemm_ms) / 1e3
    achieved = flops / gemm_s / 1e12
    whole = flops / (dev_s / args.steps) / 1e12
    launches = 2 if (A or wl.BS) else 0  # the prep kernel (codes and scale atoms), then the GEMM
    line = {
        "metric": MX_METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dev_s_max * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.mx_qtype,
        "data": "synthetic (seeded routing and N(0,1) tensors, mx-quantised per 32 along K; no dataset)",
        "config": {"workload": wl.name + "_mx_" + args.mx_qtype, "tiles": mx_tiles, "W": wl.W, "e": wl.e, "A": A,
                   "H1": wl.H1,
                   "N1": wl.N1, "BS": wl.BS, "H2": wl.H2, "N2": wl.N2, "accumulate": "fp32", "out": "bf16",
                   "l2": f"inputs rotated over {reps} replicas ({reps * nbytes / 2**20:.0f} MiB > 129 MiB L2)"},
        "timing": {
            "us_per_call_median": round(statistics.median(per_call_ms) * 1e3, 2),
            "us_per_call_min": round(min(per_call_ms) * 1e3, 2),
            "us_per_call_p90": round(float(np.percentile(per_call_ms, 90)) * 1e3, 2),
            "gemm_kernel_us_mean": round(gemm_s * 1e6, 2),
            "gemm_kernel_us_p90": round(float(np.percentile(gemm_ms, 90)) * 1e3, 2),
            "pct_of_fp8_peak": round(100 * tflops / world / peak, 2),
            "gflop_per_call": round(flops / 1e9, 3),
            "launches_per_call": launches,
        },
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(wl.name + "_mx_" + args.mx_qtype, tiles=mx_tiles,
                                                 kernel="grouped_gemm_mx_kernel"),
                     "kernel": "grouped_gemm_mx_kernel",
                     "timed": ("the GEMM kernel alone: CUDA events recorded on its launching stream right before "
                               f"and after it, mean of {args.steps} launches (a2av_gmm_mx_run_profiled)"),
                     "whole_call": {"achieved": round(whole, 2), "frac": round(whole / peak, 4),
                                    "timed": "scan + prep (codes and scale atoms) + GEMM, CUDA events around each call"},
                     "peak_source": f"2 x {pk_kind} bf16 dense burst (nominal FP8:bf16 ratio 4.5:2.25)",
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes": nbytes},
        "e2e": {"value": round(e2e_tflops, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "inputs_copied": "activation codes and scales, recvCounts, mmX codes and scales (weights resident)",
                "overlap": "step i+1's H2D and step i's D2H run on copy streams beside step i's kernels"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        f, sec, _, threads, desc = mx_oracle_sample(wl, inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(f / sec / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle", "sample": desc, "seconds": round(sec, 2)}
    emit(line)
    barrier(world)


# The process's standard output as opened at start: it carries exactly one
# JSON line.  main() points file descriptor 1 at stderr, so that whatever a
# library prints there (NCCL's version banner, for one) stays off it.
_JSON_OUT = None


def emit(obj):
    out = _JSON_OUT if _JSON_OUT is not None else sys.stdout
    out.write(json.dumps(obj) + "\n")
    out.flush()


def claim_stdout():
    """Keep the process's stdout for emit() and point file descriptor 1 at stderr."""
    global _JSON_OUT
    if _JSON_OUT is None:
        sys.stdout.flush()
        _JSON_OUT = os.fdopen(os.dup(1), "w")
        os.dup2(2, 1)


def main(argv=None):
    claim_stdout()
    os.environ.setdefault("NCCL_DEBUG_FILE", "/dev/stderr")
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--permute-out", action="store_true")
    ap.add_argument("--path", default="default", choices=["default", "fused", "split", "split_runs"])
    ap.add_argument("--tiles", default="default", choices=["default", "single", "pair", "pair_k64"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sim-rank", type=int, default=None,
                    help="N=1: time the inputs of this expert-parallel rank of the workload (default: rank 0)")
    ap.add_argument("--mx-qtype", default="e4m3fn", choices=["e4m3fn", "e5m2"], help="--op mx: code format")
    ap.add_argument("--op", default="gemm", choices=["gemm", "amp", "qreduce", "layer", "mx", "arrivals"],
                    help="gemm: the hot path (default); amp: the loss-scale step; qreduce: the quantised "
                         "rank reduce; layer: AlltoAllv + the hot path; mx: the hot path in block-scaled FP8")
    ap.add_argument("--overlap", action="store_true",
                    help="--op layer: run the shared expert beside the row exchange (default: with the routed experts)")
    ap.add_argument("--qworkload", default="qreduce_mx_e4m3_w8_rows1536_h7168",
                    help="workload of --op qreduce")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sustained-s", type=float, default=1.0,
                    help="seconds of back-to-back calls for the sustained figures (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.op == "qreduce":
        run_qreduce(args)
    elif args.op == "layer":
        run_layer(args)
    elif args.op == "mx":
        run_mx(args)
    elif args.op == "arrivals":
        run_arrivals(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.op == "amp":
        run_amp(args)
    else:
        run_gpu(args)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
