"""Throughput of the block-scaled GEMM hot path on GB300.

Default workload (the pages' published one): the atrex-bench #002
block_scaled_mm Shapes-table sweep, n=k=2048 with m in {349, 4533, 65536,
704512} and n=k=4096 with m in {237, 4096, 65536, 299520}.  One step runs the
whole hot path for all eight problems on inputs already in HBM: quantize the
float32 activations per 1x128 block, quantize the float32 weights per
128x128 block, and the FP32-scale GEMM.  Metric: TFLOPS = sum(2mnk) / step
time.  Other workloads (--workload) are the remaining configurations:
small block_scaled_mm, int8 per-channel, mxfp8, nvfp4, mxfp8 backward.

Prints one JSON line (rank 0).  With --impl reference the CPU oracle runs a
bounded sample of the same workload on the host cores instead.
Multi-GPU runs (torchrun) are independent replicas: each rank runs the full
workload on its own GPU; time is the max over ranks, value the sum of all
ranks' work over that time.
"""

from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- #
# distributed plumbing (replicas: barrier and max over ranks only)            #
# --------------------------------------------------------------------------- #

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- #
# peaks and clocks                                                            #
# --------------------------------------------------------------------------- #

def load_peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        def num(x):
            try:
                return float(x.strip())
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# --------------------------------------------------------------------------- #
# workloads on the GPU                                                        #
# --------------------------------------------------------------------------- #

class GroupedSweep:
    """block_scaled_mm problems: raw float32 a [m,k], b [n,k] resident in HBM;
    a step quantizes both and runs the FP32-scale GEMM for every problem."""
    dominant = "block-scaled FP32-scale GEMM (tc_gemm kF32Scale)"

    def __init__(self, workload: W.Workload, device):
        import block_scaled_precision_gemm_gb300 as bsmm
        self.bsmm = bsmm
        self.w = workload
        self.dev = device
        self.items = []
        for p in workload.problems:
            a_raw, b_raw = W.grouped_raw(p, workload.seed, device)
            it = {
                "p": p, "a_raw": a_raw, "b_raw": b_raw,
                "aq": torch.empty((p.m, p.k), dtype=torch.uint8, device=device),
                "sa": torch.empty((p.m, p.k // p.group_k), dtype=torch.float32, device=device),
                "bq": torch.empty((p.n, p.k), dtype=torch.uint8, device=device),
                "sb": torch.empty((p.n // p.group_n, p.k // p.group_k), dtype=torch.float32, device=device),
                "y": torch.empty((p.m, p.n), dtype=torch.float32, device=device),
            }
            self.items.append(it)
        self.flops = sum(2.0 * it["p"].m * it["p"].n * it["p"].k for it in self.items)
        self.launches_per_step = 3 * len(self.items)

    def step(self, gemm_events=None):
        b = self.bsmm
        for it in self.items:
            p = it["p"]
            b.quantize(it["a_raw"], (1, p.group_k), "e4m3", "f32", codes=it["aq"], scales=it["sa"])
            b.quantize(it["b_raw"], (p.group_n, p.group_k), "e4m3", "f32", codes=it["bq"], scales=it["sb"])
            if gemm_events is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            b.gemm_grouped(it["aq"], it["bq"], it["sa"], it["sb"], p.group_n, p.group_k, y=it["y"])
            if gemm_events is not None:
                e1.record()
                gemm_events.append((e0, e1, 2.0 * p.m * p.n * p.k))

    # ---- end to end through host buffers
    def setup_host(self):
        max_in = max(it["a_raw"].numel() + it["b_raw"].numel() for it in self.items)
        max_out = max(it["y"].numel() for it in self.items)
        self.h_in = torch.empty(max_in, dtype=torch.float32, pin_memory=True)
        self.h_out = torch.empty(max_out, dtype=torch.float32, pin_memory=True)
        # the host buffer holds real inputs (the largest problem's raw a and b)
        big = max(self.items, key=lambda it: it["a_raw"].numel())
        na = big["a_raw"].numel()
        self.h_in[:na].copy_(big["a_raw"].view(-1))
        self.h_in[na:na + big["b_raw"].numel()].copy_(big["b_raw"].view(-1))
        self.h2d = sum(4 * (it["a_raw"].numel() + it["b_raw"].numel()) for it in self.items)
        self.d2h = sum(4 * it["y"].numel() for it in self.items)

    def step_e2e(self):
        for it in self.items:
            na, nb = it["a_raw"].numel(), it["b_raw"].numel()
            it["a_raw"].view(-1).copy_(self.h_in[:na], non_blocking=True)
            it["b_raw"].view(-1).copy_(self.h_in[na:na + nb], non_blocking=True)
        self.step()
        for it in self.items:
            self.h_out[:it["y"].numel()].copy_(it["y"].view(-1), non_blocking=True)


def run_gpu(args):
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    import block_scaled_precision_gemm_gb300 as bsmm
    bsmm.lib()

    workload = selected_workload(args)
    wl = GroupedSweep(workload, device)
    torch.cuda.synchronize()

    for i in range(args.warmup):
        t0 = time.perf_counter()
        wl.step()
        if args.trace:
            torch.cuda.synchronize()
            print(f"warm-up step {i}: {1e3 * (time.perf_counter() - t0):.2f} ms", file=sys.stderr, flush=True)
    torch.cuda.synchronize()
    st, site = bsmm.check_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (site {site}) after warm-up")

    gemm_events = []
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record()
        for _ in range(args.steps):
            wl.step(gemm_events)
        e_end.record()
        torch.cuda.synchronize()
        barrier(world)
    elapsed_ms = e_start.elapsed_time(e_end)
    st, site = bsmm.check_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (site {site}) in the timed region")
    gemm_ms = sum(a.elapsed_time(b) for a, b, _ in gemm_events)
    gemm_flops = sum(f for _, _, f in gemm_events)

    t_max_ms = max_over_ranks(elapsed_ms, world, device)
    total_flops = sum_over_ranks(wl.flops * args.steps, world, device)
    value = total_flops / (t_max_ms * 1e-3) / 1e12

    # end to end: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        wl.setup_host()
        for _ in range(2):
            wl.step_e2e()
        torch.cuda.synchronize()
        barrier(world)
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(e2e_steps):
            wl.step_e2e()
        b.record()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b), world, device)
        e2e_val = sum_over_ranks(wl.flops * e2e_steps, world, device) / (e2e_ms * 1e-3) / 1e12
        e2e = {"value": round(e2e_val, 3), "unit": "TFLOPS", "h2d_bytes_per_step": wl.h2d,
               "d2h_bytes_per_step": wl.d2h, "steps": e2e_steps}

    peaks, peak_src = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops_sustained"]
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    roofline = {"kernel": wl.dominant, "bound": "tensor", "achieved": round(achieved, 2),
                "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                "traffic": TRAFFIC_PER_LAUNCH.get(args.workload),
                "peak_source": f"{peak_src}: 2 x bf16_tflops_sustained (FP8/BF16 nominal ratio 2)",
                "gemm_share_of_step": round(gemm_ms / elapsed_ms, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(workload, min_seconds=args.cpu_seconds)

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": "block-scaled GEMM TFLOPS (2MNK/t) and % of GB300 dense FP8/FP4 tensor peak",
            "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_max_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (f32 accumulate)",
            "data": "synthetic (seeded randn, the atrex-bench input recipe)",
            "config": {"workload": workload.name,
                       "problems": [[p.m, p.n, p.k] for p in workload.problems],
                       "group_n": 128, "group_k": 128,
                       "step": "quantize a 1x128 + quantize b 128x128 + FP32-scale GEMM, every problem",
                       "l2": "inputs larger than L2 (raw float32 activations %.1f GB per step)" % (
                           sum(it["a_raw"].numel() * 4 for it in wl.items) / 1e9),
                       "parallelism": f"replicas x{world}"},
            "pct_of_fp8_peak": round(100 * value / fp8_peak, 2),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": wl.launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# DRAM bytes per GEMM launch from ncu (see profiles/); None until captured
# for the kernel as it stands.
TRAFFIC_PER_LAUNCH = {}


# --------------------------------------------------------------------------- #
# CPU oracle: baseline leg and the reference arm                              #
# --------------------------------------------------------------------------- #

def oracle_sample_step(workload: W.Workload, rows: int):
    """One bounded sample of the workload on the CPU oracle: for every
    problem, the first ``rows`` activation rows against the first weight
    group (128 output columns): quantize a and b, then the grouped matmul.
    Returns the sample's FLOPs."""
    from oracle import formats as F
    from oracle import gemm as G
    from oracle import quantize as Q
    flops = 0.0
    for p in workload.problems:
        r = min(rows, p.m)
        g = torch.Generator().manual_seed(p.m)
        a = torch.randn(r, p.k, generator=g).numpy()
        b = torch.randn(p.group_n, p.k, generator=g).numpy()
        ca, sa = Q.quantize(a, (1, p.group_k), "e4m3", "f32")
        cb, sb = Q.quantize(b, (p.group_n, p.group_k), "e4m3", "f32")
        G.grouped_matmul(F.decode(ca, "e4m3"), F.decode(cb, "e4m3"), sa, sb, p.group_n, p.group_k)
        flops += 2.0 * r * p.group_n * p.k
    return flops


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload: W.Workload, min_seconds: float = 10.0, rows: int = 256):
    flops, t0 = 0.0, time.perf_counter()
    n = 0
    while True:
        flops += oracle_sample_step(workload, rows)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} passes of: first {rows} activation rows x first 128 output columns of each of the "
                      f"{len(workload.problems)} problems (quantize a, quantize b, grouped matmul; NumPy float64)",
            "seconds": round(el, 2)}


def selected_workload(args) -> W.Workload:
    if args.problem:
        m, n, k = (int(v) for v in args.problem.split(","))
        return W.Workload(f"block_scaled_mm m={m} n={n} k={k}", W.GROUPED_SWEEP.seed, (W.Grouped(m, n, k),))
    return WORKLOADS_BY_KEY[args.workload]


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    workload = selected_workload(args)
    rows = args.reference_rows
    for _ in range(args.warmup):
        oracle_sample_step(workload, rows)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_sample_step(workload, rows)
    el = time.perf_counter() - t0
    value = flops / el / 1e12
    sample = (f"first {rows} activation rows x first 128 output columns of each of the "
              f"{len(workload.problems)} problems per step")
    line = {
        "impl": "reference",
        "metric": "block-scaled GEMM TFLOPS (2MNK/t) and % of GB300 dense FP8/FP4 tensor peak",
        "value": round(value, 6), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded randn, the atrex-bench input recipe)",
        "config": {"workload": workload.name, "problems": [[p.m, p.n, p.k] for p in workload.problems],
                   "group_n": 128, "group_k": 128, "sample": sample},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


WORKLOADS_BY_KEY = {"sweep": W.GROUPED_SWEEP, "small": W.GROUPED_SMALL}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS_BY_KEY), default="sweep")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-rows", type=int, default=64)
    ap.add_argument("--problem", default=None, help="one block_scaled_mm problem 'm,n,k' instead of --workload")
    ap.add_argument("--trace", action="store_true", help="print warm-up step times to stderr")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
