"""Throughput of the block-scaled GEMM hot path on GB300.

Default workload (the pages' published one): the atrex-bench #002
block_scaled_mm Shapes-table sweep, n=k=2048 with m in {349, 4533, 65536,
704512} and n=k=4096 with m in {237, 4096, 65536, 299520}.  One step runs the
whole hot path for all eight problems on inputs already in HBM: quantize the
float32 activations per 1x128 block, quantize the float32 weights per
128x128 block, and the FP32-scale GEMM.  Metric: TFLOPS = sum(2mnk) / step
time.  Other workloads (--workload) are the remaining configurations:
small block_scaled_mm, int8 per-channel, mxfp8, nvfp4, mxfp8 backward, and mxfp4 (the
next format, at the nvfp4 size).

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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
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
    """nvidia-smi sampling of SM clocks and throttle reasons.

    A reader thread stamps each sample with the host clock when it arrives, so
    that the summary can keep the samples of one window (the timed region).
    Entering waits for the first sample, so the sampler is live before the
    window opens."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.thread = None
        self.rows = []  # (host time of arrival, csv fields)
        self.window = (float("-inf"), float("inf"))
        self.note = "timed region"

    def _read(self):
        for line in self.proc.stdout:
            fields = next(csv.reader([line]), [])
            if len(fields) >= 9:
                self.rows.append((time.perf_counter(), fields))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.perf_counter()
        while not self.rows and self.proc.poll() is None and time.perf_counter() - t0 < 5.0:
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def count(self, t0, t1):
        return sum(1 for t, _ in self.rows if t0 <= t <= t1)

    def set_window(self, t0, t1, note):
        self.window, self.note = (t0, t1), note

    def summary(self, window=None):
        t0, t1 = window or self.window
        rows = [r for t, r in self.rows if t0 <= t <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0,
                    "window": self.note}
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
                "reasons": reasons, "samples": len(rows), "window": self.note,
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# --------------------------------------------------------------------------- #
# workloads on the GPU                                                        #
# --------------------------------------------------------------------------- #

def _ev():
    return torch.cuda.Event(enable_timing=True)


class Work:
    """One configuration: buffers resident in HBM, a step that runs the whole
    hot path on them, its FLOPs, and an end-to-end variant through pinned host
    buffers.  ``step(events)`` appends (start, end, flops) around every launch
    of the dominant call."""
    peak_kind = "fp8"
    dtype = "e4m3 (f32 accumulate)"

    def quantizer_bytes(self):
        """[(label, kernel name, algorithmic bytes per launch)] for the step's
        quantizer launches, in launch order (a name that repeats is matched
        in turn; a trailing * matches any kernel with that prefix); empty
        where the step has none.  A list of such lists gives alternatives
        (the library picks kernels by shape and alignment): the first whose
        kernels all ran is used."""
        return []

    @staticmethod
    def _matches(n, kname):
        return n == kname or (kname.endswith("*") and n.startswith(kname[:-1]))

    def quantizer_report(self, launches, steps):
        """Per-kernel HBM throughput of the step's quantizers from the
        library's own per-launch CUDA events (bsmm.trace over `steps` untimed
        steps), and the span from the first quantizer's start to the last
        one's end."""
        want = self.quantizer_bytes()
        if not want:
            return None
        per_step = len(launches) // steps
        if isinstance(want[0], list):  # alternatives
            first = [n for n, _, _ in launches[:per_step]]
            want = next(alt for alt in want if all(any(self._matches(n, k) for n in first) for _, k, _ in alt))
        out, spans = {}, []
        for st in range(steps):
            mine = launches[st * per_step:(st + 1) * per_step]
            used = [False] * len(mine)
            t_lo, t_hi, nbytes = None, None, 0
            for label, kname, nb in want:
                i = next(i for i, (n, _, _) in enumerate(mine) if not used[i] and self._matches(n, kname))
                used[i] = True
                n, t0, ms = mine[i]
                e = out.setdefault(label, {"kernel": n, "ms": 0.0, "bytes": 0})
                e["ms"] += ms
                e["bytes"] += nb
                t_lo = t0 if t_lo is None else min(t_lo, t0)
                t_hi = t0 + ms if t_hi is None else max(t_hi, t0 + ms)
                nbytes += nb
            spans.append((t_hi - t_lo, nbytes))
        rep = {}
        for label, e in out.items():
            rep[label] = {"kernel": e["kernel"], "gbs": round(e["bytes"] / (e["ms"] * 1e-3) / 1e9, 1),
                          "us_per_step": round(1e3 * e["ms"] / steps, 2), "bytes_per_step": int(e["bytes"] / steps)}
        if len(want) > 1:
            ms = sum(t for t, _ in spans)
            nb = sum(b for _, b in spans)
            rep["all quantizers, first start to last end"] = {
                "gbs": round(nb / (ms * 1e-3) / 1e9, 1), "us_per_step": round(1e3 * ms / steps, 2),
                "bytes_per_step": int(nb / steps)}
        return rep

    def _timed(self, events, flops, fn):
        if events is None:
            return fn()
        e0, e1 = _ev(), _ev()
        e0.record()
        r = fn()
        e1.record()
        events.append((e0, e1, flops))
        return r

    def setup_host(self):
        self.h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in self.inputs]
        self.h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in self.outputs]
        self.h2d = sum(t.numel() * t.element_size() for t in self.inputs)
        self.d2h = sum(t.numel() * t.element_size() for t in self.outputs)

    def step_e2e(self):
        for d, h in zip(self.inputs, self.h_in):
            d.copy_(h, non_blocking=True)
        self.step()
        for d, h in zip(self.outputs, self.h_out):
            h.copy_(d, non_blocking=True)


class GroupedWork(Work):
    """block_scaled_mm problems: raw float32 a [m,k], b [n,k] in HBM; a step
    quantizes both (1x128, 128x128) and runs the FP32-scale GEMM."""
    dominant = "block-scaled FP32-scale GEMM (tc_gemm_pair kPairF32; tc_gemm kF32Scale below one tile per cluster)"

    def __init__(self, workload: W.Workload, device):
        import block_scaled_precision_gemm_gb300 as bsmm
        self.bsmm, self.w = bsmm, workload
        self.items = []
        for p in workload.problems:
            a_raw, b_raw = W.grouped_raw(p, workload.seed, device)
            self.items.append({
                "p": p, "a_raw": a_raw, "b_raw": b_raw,
                "aq": torch.empty((p.m, p.k), dtype=torch.uint8, device=device),
                "sa": torch.empty((p.m, p.k // p.group_k), dtype=torch.float32, device=device),
                "bq": torch.empty((p.n, p.k), dtype=torch.uint8, device=device),
                "sb": torch.empty((p.n // p.group_n, p.k // p.group_k), dtype=torch.float32, device=device),
                "y": torch.empty((p.m, p.n), dtype=torch.float32, device=device)})
        self.flops = sum(2.0 * it["p"].m * it["p"].n * it["p"].k for it in self.items)
        # every problem's weight quantization in one call (its 128 x 128 tiles share launches)
        self.b_jobs = [{"x": it["b_raw"], "block": (it["p"].group_n, it["p"].group_k), "code": "e4m3", "scale": "f32",
                        "codes": it["bq"], "scales": it["sb"]} for it in self.items]
        self.inputs = [t for it in self.items for t in (it["a_raw"], it["b_raw"])]
        self.outputs = [it["y"] for it in self.items]

    def step(self, events=None):
        b = self.bsmm
        b.quantize_batch(self.b_jobs)
        for it in self.items:
            p = it["p"]
            b.quantize(it["a_raw"], (1, p.group_k), "e4m3", "f32", codes=it["aq"], scales=it["sa"])
            self._timed(events, 2.0 * p.m * p.n * p.k, lambda: b.gemm_grouped(
                it["aq"], it["bq"], it["sa"], it["sb"], p.group_n, p.group_k, y=it["y"]))

    def quantizer_bytes(self):
        # algorithmic bytes: float32 read, one code byte and the scales written
        out = [("quant_tile_batch (b, 128x128, every problem's weight in one launch)", "quant_tile_batch",
                sum(4 * it["p"].n * it["p"].k + it["p"].n * it["p"].k +
                    4 * (it["p"].n // it["p"].group_n) * (it["p"].k // it["p"].group_k) for it in self.items))]
        for it in self.items:
            p = it["p"]
            out.append(("quant_rows (a, 1x128)", "quant_rows", 4 * p.m * p.k + p.m * p.k + 4 * p.m * (p.k // p.group_k)))
        return out

    def quantizer_report(self, launches, steps):
        rep = Work.quantizer_report(self, launches, steps)
        rep.pop("all quantizers, first start to last end", None)  # the GEMMs run between them
        return rep

    def setup_host(self):
        # one pinned buffer per direction, sized for the largest problem, reused
        # by every problem (the copies are the step's real traffic)
        max_in = max(it["a_raw"].numel() + it["b_raw"].numel() for it in self.items)
        max_out = max(it["y"].numel() for it in self.items)
        self.hb_in = torch.empty(max_in, dtype=torch.float32, pin_memory=True)
        self.hb_out = torch.empty(max_out, dtype=torch.float32, pin_memory=True)
        big = max(self.items, key=lambda it: it["a_raw"].numel())
        na = big["a_raw"].numel()
        self.hb_in[:na].copy_(big["a_raw"].view(-1))
        self.hb_in[na:na + big["b_raw"].numel()].copy_(big["b_raw"].view(-1))
        self.h2d = sum(4 * (it["a_raw"].numel() + it["b_raw"].numel()) for it in self.items)
        self.d2h = sum(4 * it["y"].numel() for it in self.items)

    E2E_ROWS = 65536  # activation rows per pipelined chunk

    def step_e2e(self):
        """The same step from pinned host buffers, pipelined over row chunks of
        each problem on three streams: copy in, compute, copy out.  Each row's
        quantization and output depend on that row alone, so the chunked
        calls give exactly the unchunked results."""
        b = self.bsmm
        cur = torch.cuda.current_stream()
        if not hasattr(self, "s_in"):
            self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        s_in, s_out = self.s_in, self.s_out
        s_in.wait_stream(cur)   # the previous step has finished reading the inputs
        cur.wait_stream(s_out)  # ... and copying the outputs out
        for it in self.items:
            p = it["p"]
            na, nb = it["a_raw"].numel(), it["b_raw"].numel()
            with torch.cuda.stream(s_in):
                it["b_raw"].view(-1).copy_(self.hb_in[na:na + nb], non_blocking=True)
            for r0 in range(0, p.m, self.E2E_ROWS):
                r1 = min(p.m, r0 + self.E2E_ROWS)
                lo, hi = r0 * p.k, r1 * p.k
                with torch.cuda.stream(s_in):
                    it["a_raw"].view(-1)[lo:hi].copy_(self.hb_in[lo:hi], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record()
                cur.wait_event(ev_in)
                if r0 == 0:
                    b.quantize(it["b_raw"], (p.group_n, p.group_k), "e4m3", "f32", codes=it["bq"], scales=it["sb"])
                b.quantize(it["a_raw"][r0:r1], (1, p.group_k), "e4m3", "f32", codes=it["aq"][r0:r1],
                           scales=it["sa"][r0:r1])
                b.gemm_grouped(it["aq"][r0:r1], it["bq"], it["sa"][r0:r1], it["sb"], p.group_n, p.group_k,
                               y=it["y"][r0:r1])
                ev_c = torch.cuda.Event()
                ev_c.record()
                s_out.wait_event(ev_c)
                with torch.cuda.stream(s_out):
                    self.hb_out[r0 * p.n:r1 * p.n].copy_(it["y"][r0:r1].view(-1), non_blocking=True)
        cur.wait_stream(s_out)

    def config(self):
        return {"problems": [[p.m, p.n, p.k] for p in self.w.problems], "group_n": 128, "group_k": 128,
                "step": "quantize a 1x128 + quantize b 128x128 + FP32-scale GEMM, every problem"}

    def input_bytes(self):
        return sum(it["a_raw"].numel() * 4 for it in self.items)


class Int8Work(Work):
    """TensorTonic INT8 per-channel matmul at B = D_in = D_out = 4096: a step
    quantizes x per row and w per column and runs the exact int32 matmul."""
    dominant = "INT8 per-channel call (quantizers + tc_gemm_pair kPairI8: exact int sums on bf16 tensor cores)"
    peak_kind = "int8"
    dtype = "int8 (int32 accumulate)"

    def __init__(self, workload, device):
        import block_scaled_precision_gemm_gb300 as bsmm
        self.bsmm, self.w = bsmm, workload
        self.p = p = workload.problems[0]
        self.x, self.wt = W.int8_raw(p, workload.seed, device)
        self.out = {"x_q": torch.empty((p.B, p.D_in), dtype=torch.int8, device=device),
                    "x_scales": torch.empty(p.B, dtype=torch.float32, device=device),
                    "w_q": torch.empty((p.D_in, p.D_out), dtype=torch.int8, device=device),
                    "w_scales": torch.empty(p.D_out, dtype=torch.float32, device=device),
                    "y": torch.empty((p.B, p.D_out), dtype=torch.float32, device=device)}
        self.ws = torch.empty(bsmm.int8_channel_workspace_size(p.B, p.D_in, p.D_out), dtype=torch.uint8,
                              device=device)
        self.flops = 2.0 * p.B * p.D_in * p.D_out
        self.inputs, self.outputs = [self.x, self.wt], [self.out["y"]]

    def step(self, events=None):
        self._timed(events, self.flops, lambda: self.bsmm.int8_channel(self.x, self.wt, out=self.out,
                                                                      workspace=self.ws))

    def quantizer_bytes(self):
        # float32 read, int8 codes, the matmul's zero-padded bf16 copy, FP32 scales
        p = self.p
        Kp = -(-p.D_in // 128) * 128
        w_bytes = 4 * p.D_in * p.D_out + p.D_in * p.D_out + 2 * p.D_out * Kp + 4 * p.D_out
        x_bytes = 4 * p.B * p.D_in + p.B * p.D_in + 2 * p.B * Kp + 4 * p.B
        return [("w per column (second stream)", "i8_quant_w_*", w_bytes), ("x per row", "i8_quant_rows*", x_bytes)]

    def config(self):
        p = self.p
        return {"B": p.B, "D_in": p.D_in, "D_out": p.D_out, "zero_frac": p.zero_frac,
                "step": "x per-row + w per-column INT8 quantize, int32 matmul, y = a*sx*sw"}

    def input_bytes(self):
        return 4 * (self.x.numel() + self.wt.numel())


class MxWork(Work):
    """jax.nn.scaled_matmul with the Blackwell formats: MXFP8 B=8,
    M=N=4096, K=8192 or NVFP4 B=1, M=N=K=16384.  Codes and scales are
    resident; a step is the library call (scale relayout + GEMM)."""

    def __init__(self, workload, device):
        import block_scaled_precision_gemm_gb300 as bsmm
        self.bsmm, self.w = bsmm, workload
        self.p = p = workload.problems[0]
        raw = W.batched_raw(p, workload.seed, device)
        if p.fmt == "mxfp8":
            # encoding the seeded draws is input preparation (torch's float8 cast)
            self.a = raw[0].to(torch.float8_e4m3fn).view(torch.uint8)
            self.b = raw[1].to(torch.float8_e4m3fn).view(torch.uint8)
            self.sa = (raw[2] + 127).to(torch.uint8)
            self.sb = (raw[3] + 127).to(torch.uint8)
            self.types = ("e4m3", "e4m3", "ue8m0")
            self.dominant = "MXFP8 block-scaled GEMM call (sf_relayout + tc_gemm_pair kPairMXF8)"
        elif p.fmt == "mxfp4":
            self.a, self.b = raw[0], raw[1]
            self.sa = (raw[2] + 127).to(torch.uint8)
            self.sb = (raw[3] + 127).to(torch.uint8)
            self.types = ("e2m1", "e2m1", "ue8m0")
            self.peak_kind = "fp4"
            self.dtype = "e2m1 (f32 accumulate)"
            self.dominant = "MXFP4 block-scaled GEMM call (sf_relayout + tc_gemm_pair kPairMXF4)"
        else:
            self.a, self.b = raw[0], raw[1]
            self.sa = raw[2].to(torch.float8_e4m3fn).view(torch.uint8)
            self.sb = raw[3].to(torch.float8_e4m3fn).view(torch.uint8)
            self.types = ("e2m1", "e2m1", "ue4m3")
            self.peak_kind = "fp4"
            self.dtype = "e2m1 (f32 accumulate)"
            self.dominant = "NVFP4 block-scaled GEMM call (sf_relayout + tc_gemm_pair kPairNVF4)"
        del raw
        self.y = torch.empty((p.B, p.M, p.N), dtype=torch.float32, device=device)
        self.ws = torch.empty(bsmm.gemm_workspace_size(p.B, p.M, p.N, p.K, self.types[0]), dtype=torch.uint8,
                              device=device)
        self.flops = 2.0 * p.B * p.M * p.N * p.K
        self.inputs, self.outputs = [self.a, self.b, self.sa, self.sb], [self.y]

    def step(self, events=None):
        t = self.types
        self._timed(events, self.flops, lambda: self.bsmm.gemm(self.a, self.b, self.sa, self.sb, t[0], t[1], t[2],
                                                               y=self.y, workspace=self.ws, K=self.p.K))

    def config(self):
        p = self.p
        return {"B": p.B, "M": p.M, "N": p.N, "K": p.K, "format": p.fmt,
                "step": "scale relayout + block-scaled GEMM, FP32 output"}

    def input_bytes(self):
        return sum(t.numel() for t in self.inputs)


class BackwardWork(Work):
    """NKI MXFP8 linear backward, M=16384, N=K=8192: a step quantizes dY (along
    N and along M), W (along N) and X (along M) to E5M2 and runs dX = dY.W and
    dW = dY^T.X with bf16 outputs."""
    dominant = "MXFP8 backward call (dual dY quantizer + W^T, X^T quantizers into scale atoms + 2 x tc_gemm_pair kPairMXF8)"
    dtype = "e5m2 (f32 accumulate, bf16 out)"

    def __init__(self, workload, device):
        import block_scaled_precision_gemm_gb300 as bsmm
        self.bsmm, self.w = bsmm, workload
        self.p = p = workload.problems[0]
        self.dY, self.W, self.X = W.backward_raw(p, workload.seed, device)
        self.dX = torch.empty((p.M, p.K), dtype=torch.bfloat16, device=device)
        self.dW = torch.empty((p.N, p.K), dtype=torch.bfloat16, device=device)
        self.ws = torch.empty(bsmm.linear_backward_workspace_size(p.M, p.N, p.K), dtype=torch.uint8,
                              device=device)
        self.flops = 2 * 2.0 * p.M * p.N * p.K
        self.inputs, self.outputs = [self.dY, self.W, self.X], [self.dX, self.dW]

    def step(self, events=None):
        self._timed(events, self.flops, lambda: self.bsmm.linear_backward(
            self.dY, self.W, self.X, self.p.fp8, dX=self.dX, dW=self.dW, workspace=self.ws))

    def _quantized_operands(self):
        """The four operands the call leaves in its workspace, in the order and
        alignment the header documents: codes, then atoms, each part on a
        256-byte boundary."""
        p, ws, out, off = self.p, self.ws, [], 0
        for rows, cols in ((p.M, p.N), (p.K, p.N), (p.N, p.M), (p.K, p.M)):
            codes = ws[off:off + rows * cols].view(rows, cols)
            off += -(-rows * cols // 256) * 256
            n = self.bsmm.scale_atoms_size(1, rows, cols, p.fp8, "ue8m0")
            out += [codes, ws[off:off + n]]
            off += -(-n // 256) * 256
        return out

    def quantizer_bytes(self):
        # bf16 read once, E5M2 codes and UE8M0 scales (one per 32) written
        p = self.p
        M, N, K = p.M, p.N, p.K
        dual = ("quant_cols_tma2 dual (dY along N and along M)", "quant_cols_tma2 (dual)",
                2 * M * N + 2 * (M * N + M * N // 32))
        wt, xt = 2 * N * K + N * K + N * K // 32, 2 * M * K + M * K + M * K // 32
        return [[dual, ("quant_cols_tma2 pair (W along N -> W^T and X along M -> X^T)", "quant_cols_tma2 (pair)",
                        wt + xt)],
                [dual, ("quant_cols_tma2 (W along N -> W^T)", "quant_cols_tma2", wt),
                 ("quant_cols_tma2 (X along M -> X^T)", "quant_cols_tma2", xt)]]

    def config(self):
        p = self.p
        return {"M": p.M, "N": p.N, "K": p.K, "fp8": p.fp8,
                "step": "4 MXFP8 quantizers + dX = dY.W and dW = dY^T.X, bf16 outputs"}

    def input_bytes(self):
        return sum(t.numel() * 2 for t in self.inputs)


def make_work(workload: W.Workload, device) -> Work:
    p = workload.problems[0]
    if isinstance(p, W.Grouped):
        return GroupedWork(workload, device)
    if isinstance(p, W.Int8Channel):
        return Int8Work(workload, device)
    if isinstance(p, W.Batched):
        return MxWork(workload, device)
    return BackwardWork(workload, device)


def peak_tflops(peaks, kind, sustained):
    """Dense peak for the path's own dtype: measured bf16 times the nominal
    dense ratio on GB300 (FP8 4.5/2.25 = 2x, FP4 13.5/2.25 = 6x).  INT8 has no
    measured or usable nominal figure on this part: its exact matmul runs on
    the bf16 tensor cores, so the bf16 rate is its peak.

    ``sustained`` picks the bf16 figure measured back to back under the power
    cap, for a timed region that ran under it; otherwise the burst figure."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    base = peaks[key]
    return {"fp8": 2.0 * base, "fp4": 6.0 * base, "int8": base}[kind], {
        "fp8": f"2 x {key} (FP8/BF16 nominal dense ratio 4.5/2.25)",
        "fp4": f"6 x {key} (FP4/BF16 nominal dense ratio 13.5/2.25)",
        "int8": f"{key} (the INT8 matmul runs exactly on the bf16 tensor cores)"}[kind]


SUSTAINED_REGION_S = 2.0


def use_sustained_peak(clocks, region_s):
    """The sustained bf16 figure was measured back to back for seconds under
    the power cap; it is the denominator only for a timed region that is
    itself seconds long and ran under the cap (sw_power_cap active).  A
    shorter region is a burst, whatever the sampler saw."""
    return region_s >= SUSTAINED_REGION_S and "sw_power_cap" in clocks.get("reasons", [])


def measure(workload, args, device, rank, world, local, cpu_seconds):
    """Runs one workload: warm-up, the timed region (CUDA events on the
    launching stream, clocks sampled), the end-to-end leg, the CPU oracle
    leg.  Returns the record's fields (rank 0 prints them)."""
    import block_scaled_precision_gemm_gb300 as bsmm
    wl = make_work(workload, device)
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

    events = []
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t_open = time.perf_counter()
        e_start, e_end = _ev(), _ev()
        e_start.record()
        for _ in range(args.steps):
            wl.step(events)
        e_end.record()
        torch.cuda.synchronize()
        t_close = time.perf_counter()
        clk.set_window(t_open, t_close, "timed region")
        region = (t_open, t_close)
        if clk.count(t_open, t_close) < 3:
            # a timed region shorter than a few sampling periods: the clocks
            # are those of further, untimed steps of the same workload run
            # straight after it (at most two seconds of them)
            while clk.count(t_open, time.perf_counter()) < 3 and time.perf_counter() - t_close < 2.0:
                for _ in range(args.steps):
                    wl.step()
                torch.cuda.synchronize()
            clk.set_window(t_open, time.perf_counter(),
                           f"timed region ({1e3 * (t_close - t_open):.0f} ms) and the untimed steps of the same "
                           "workload run right after it")
        barrier(world)
    elapsed_ms = e_start.elapsed_time(e_end)
    st, site = bsmm.check_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (site {site}) in the timed region")
    dom_ms = sum(a.elapsed_time(b) for a, b, _ in events)
    dom_flops = sum(f for _, _, f in events)

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
        a, b = _ev(), _ev()
        a.record()
        for _ in range(e2e_steps):
            wl.step_e2e()
        b.record()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b), world, device)
        e2e_val = sum_over_ranks(wl.flops * e2e_steps, world, device) / (e2e_ms * 1e-3) / 1e12
        e2e = {"value": round(e2e_val, 3), "unit": "TFLOPS", "h2d_bytes_per_step": wl.h2d,
               "d2h_bytes_per_step": wl.d2h, "steps": e2e_steps}

    clocks = clk.summary()
    in_region = clk.summary(region)
    region_s = region[1] - region[0]
    sustained = use_sustained_peak(in_region, region_s)
    peaks, peak_src = load_peaks()
    peak, peak_how = peak_tflops(peaks, wl.peak_kind, sustained)
    capped_seen = "sw_power_cap" in in_region.get("reasons", [])
    peak_how += (f"; the {region_s:.2f} s timed region ran under the power cap" if sustained else
                 f"; a {region_s:.2f} s timed region is a burst"
                 + (" (sw_power_cap seen in it)" if capped_seen else ""))
    clocks["timed_region_samples"] = in_region["samples"]
    clocks["timed_region_reasons"] = in_region["reasons"]
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    roofline = {"kernel": wl.dominant, "bound": "tensor", "achieved": round(achieved, 2),
                "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": TRAFFIC_PER_LAUNCH.get(workload.name),
                "traffic_unit": "bytes per launch (ncu DRAM read + write)",
                "peak_source": f"{peak_src}: {peak_how}",
                "share_of_step": round(dom_ms / elapsed_ms, 4)}

    # per-kernel times from the library's own events, over a few untimed steps
    trace_steps = 3
    with bsmm.trace() as launches:
        for _ in range(trace_steps):
            wl.step()
    kernels = {}
    for name, _, ms in launches:
        k = kernels.setdefault(name, {"launches": 0, "us": 0.0})
        k["launches"] += 1
        k["us"] += 1e3 * ms
    for k in kernels.values():
        k["launches"] = k["launches"] // trace_steps
        k["us"] = round(k["us"] / trace_steps, 2)
    launches_per_step = len(launches) // trace_steps
    quant = wl.quantizer_report(launches, trace_steps)
    if quant:
        hbm = load_peaks()[0]["hbm_gbs"]
        for q in quant.values():
            q["frac_of_hbm"] = round(q["gbs"] / hbm, 3)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(workload, min_seconds=cpu_seconds)

    cfg = describe(workload)
    cfg["l2"] = "inputs larger than L2 (%.2f GB resident inputs per step)" % (wl.input_bytes() / 1e9)
    cfg["parallelism"] = f"replicas x{world}"
    rec = {
        "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max_ms / args.steps, 4), "dtype": wl.dtype,
        "config": cfg,
        "pct_of_peak": round(100 * value / peak, 2),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "kernels_per_step": {"how": "bsmm.trace: the library's CUDA events around each of its launches, mean of "
                                    f"{trace_steps} untimed steps", **kernels},
        "clocks": clocks,
    }
    if quant:
        rec["quantizers"] = quant
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


# The default run's other configurations, each a sub-record of the headline
# line: the pages' remaining workloads and the next format (MXFP4).
SUB_CONFIGS = ("int8", "mxfp8", "nvfp4", "backward", "mxfp4")


def run_gpu(args):
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    import block_scaled_precision_gemm_gb300 as bsmm
    bsmm.lib()

    head = measure(selected_workload(args), args, device, rank, world, local, args.cpu_seconds)
    subs = {}
    if args.workload is None and not args.problem and not args.headline_only:
        for key in SUB_CONFIGS:
            rec = measure(WORKLOADS_BY_KEY[key], args, device, rank, world, local, args.sub_cpu_seconds)
            if key == "mxfp4":
                rec["note"] = "next format (MXFP4: E2M1 codes, UE8M0 scale per 32), at the NVFP4 size"
            subs[key] = rec
    if rank == 0:
        line = {
            "metric": "block-scaled GEMM TFLOPS (2MNK/t) and % of GB300 dense FP8/FP4 tensor peak",
            "value": head["value"], "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
            "data": "synthetic (seeded draws with the pages' shapes and distributions)",
            "config": head["config"],
            "pct_of_peak": head["pct_of_peak"],
            "roofline": head["roofline"],
            "cpu_baseline": head["cpu_baseline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"] + sum(r["gpu_launches"] for r in subs.values()),
            "clocks": head["clocks"],
        }
        if "quantizers" in head:
            line["quantizers"] = head["quantizers"]
        if subs:
            line["gpu_launches_headline"] = head["gpu_launches"]
            line["configs"] = subs
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the dominant kernel or call, from ncu captures of the same workloads;
# None until captured for the kernels as they stand.  sweep: the mean over the step's 8 GEMM launches.  mxfp8,
# nvfp4, mxfp4: the GEMM launch (the scale relayouts add under 1%).
# backward (5 launches) and int8 (3): the whole call.
TRAFFIC_PER_LAUNCH = {
    W.GROUPED_SWEEP.name: 1_971_700_000,
    W.MXFP8_BATCHED.name: 1_317_400_000,
    W.NVFP4_SQUARE.name: 4_353_200_000,
    W.MXFP4_SQUARE.name: 2_436_300_000,
    W.BACKWARD.name: 3_233_100_000,
    W.INT8_4096.name: 317_200_000,
}


# --------------------------------------------------------------------------- #
# CPU oracle: baseline leg and the reference arm                              #
# --------------------------------------------------------------------------- #

def describe(workload: W.Workload) -> dict:
    """The configuration keys of a workload (no device needed)."""
    p = workload.problems[0]
    cfg = {"workload": workload.name}
    if isinstance(p, W.Grouped):
        cfg.update({"problems": [[q.m, q.n, q.k] for q in workload.problems], "group_n": p.group_n,
                    "group_k": p.group_k,
                    "step": "quantize a 1x128 + quantize b 128x128 + FP32-scale GEMM, every problem"})
    elif isinstance(p, W.Int8Channel):
        cfg.update({"B": p.B, "D_in": p.D_in, "D_out": p.D_out, "zero_frac": p.zero_frac,
                    "step": "x per-row + w per-column INT8 quantize, int32 matmul, y = a*sx*sw"})
    elif isinstance(p, W.Batched):
        cfg.update({"B": p.B, "M": p.M, "N": p.N, "K": p.K, "format": p.fmt,
                    "step": "scale relayout + block-scaled GEMM, FP32 output"})
    else:
        cfg.update({"M": p.M, "N": p.N, "K": p.K, "fp8": p.fp8,
                    "step": "4 MXFP8 quantizers + dX = dY.W and dW = dY^T.X, bf16 outputs"})
    return cfg


def oracle_sample(workload: W.Workload, rows: int):
    """A bounded sample of the workload for the CPU oracle.  Returns
    ``(flops, run, text)``: ``run()`` executes every step of the hot path on
    the sample (inputs are drawn beforehand, outside the timing)."""
    from oracle import formats as F
    from oracle import gemm as G
    from oracle import quantize as Q
    p = workload.problems[0]
    g = torch.Generator().manual_seed(workload.seed)
    if isinstance(p, W.Grouped):
        data = []
        for q in workload.problems:
            r = min(rows, q.m)
            data.append((q, torch.randn(r, q.k, generator=g).numpy(), torch.randn(q.group_n, q.k, generator=g).numpy()))

        def run():
            for q, a, b in data:
                ca, sa = Q.quantize(a, (1, q.group_k), "e4m3", "f32")
                cb, sb = Q.quantize(b, (q.group_n, q.group_k), "e4m3", "f32")
                G.grouped_matmul(F.decode(ca, "e4m3"), F.decode(cb, "e4m3"), sa, sb, q.group_n, q.group_k)
        flops = sum(2.0 * a.shape[0] * q.group_n * q.k for q, a, _ in data)
        text = (f"first {rows} activation rows x first 128 output columns of each of the "
                f"{len(workload.problems)} problems (quantize a, quantize b, grouped matmul)")
        return flops, run, text
    if isinstance(p, W.Int8Channel):
        r = min(rows, p.B)
        x = torch.randn(r, p.D_in, generator=g).numpy()
        w = torch.randn(p.D_in, 128, generator=g).numpy()
        return (2.0 * r * p.D_in * 128, lambda: G.int8_channel(x, w),
                f"first {r} rows of x x first 128 columns of w (both quantizers, int64 matmul, y)")
    if isinstance(p, W.Batched):
        r = min(rows, p.M)
        if p.fmt == "mxfp8":
            a = torch.randint(0, 256, (1, r, p.K), generator=g).numpy().astype(np.uint8) & 0x77
            b = torch.randint(0, 256, (1, 128, p.K), generator=g).numpy().astype(np.uint8) & 0x77
            sa = torch.randint(121, 134, (1, r, p.K // 32), generator=g).numpy().astype(np.uint8)
            sb = torch.randint(121, 134, (1, 128, p.K // 32), generator=g).numpy().astype(np.uint8)
            run = lambda: G.scaled_matmul(F.decode(a, "e4m3"), F.decode(b, "e4m3"), F.decode(sa, "ue8m0"),  # noqa
                                          F.decode(sb, "ue8m0"))
        elif p.fmt == "mxfp4":
            a = torch.randint(0, 256, (1, r, p.K // 2), generator=g).numpy().astype(np.uint8)
            b = torch.randint(0, 256, (1, 128, p.K // 2), generator=g).numpy().astype(np.uint8)
            sa = torch.randint(121, 134, (1, r, p.K // 32), generator=g).numpy().astype(np.uint8)
            sb = torch.randint(121, 134, (1, 128, p.K // 32), generator=g).numpy().astype(np.uint8)
            run = lambda: G.scaled_matmul(F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1"),  # noqa
                                          F.decode(sa, "ue8m0"), F.decode(sb, "ue8m0"))
        else:
            a = torch.randint(0, 256, (1, r, p.K // 2), generator=g).numpy().astype(np.uint8)
            b = torch.randint(0, 256, (1, 128, p.K // 2), generator=g).numpy().astype(np.uint8)
            sa = torch.randint(0x18, 0x58, (1, r, p.K // 16), generator=g).numpy().astype(np.uint8)
            sb = torch.randint(0x18, 0x58, (1, 128, p.K // 16), generator=g).numpy().astype(np.uint8)
            run = lambda: G.scaled_matmul(F.decode(F.unpack_e2m1(a), "e2m1"), F.decode(F.unpack_e2m1(b), "e2m1"),  # noqa
                                          F.decode(sa, "ue4m3"), F.decode(sb, "ue4m3"))
        return (2.0 * r * 128 * p.K, run,
                f"first {r} rows x first 128 columns of batch 0 (decode, scale, float64 matmul)")
    r = min(rows, p.M)
    dY_rows = torch.randn(r, p.N, generator=g).numpy()
    w_cols = (torch.randn(p.N, 128, generator=g) * 0.02).numpy()
    dY_cols = torch.randn(p.M, 128, generator=g).numpy()
    x_cols = (torch.randn(p.M, 128, generator=g) * 0.02).numpy()

    def run():
        # dX[:r, :128]: dY rows along N, W columns along N
        cq, cs = G.mx_quantize(dY_rows, "cols", p.fp8)
        wq, ws = G.mx_quantize(w_cols, "rows", p.fp8)
        G.scaled_matmul(F.decode(cq, p.fp8)[None], F.decode(wq, p.fp8)[None], F.decode(cs, "ue8m0")[None],
                        F.decode(ws, "ue8m0")[None])
        # dW[:128, :128]: dY columns along M, X columns along M
        dq, ds = G.mx_quantize(dY_cols, "rows", p.fp8)
        xq, xs = G.mx_quantize(x_cols, "rows", p.fp8)
        G.scaled_matmul(F.decode(dq, p.fp8)[None], F.decode(xq, p.fp8)[None], F.decode(ds, "ue8m0")[None],
                        F.decode(xs, "ue8m0")[None])
    return (2.0 * r * p.N * 128 + 2.0 * 128 * p.M * 128, run,
            f"dX[:{r}, :128] and dW[:128, :128] (all four MXFP8 quantizers on the needed lines, both matmuls)")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload: W.Workload, min_seconds: float = 10.0, rows: int = 256):
    flops_one, run, text = oracle_sample(workload, rows)
    flops, n, t0 = 0.0, 0, time.perf_counter()
    while True:
        run()
        flops += flops_one
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} passes of: {text}; NumPy float64 oracle", "seconds": round(el, 2)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    workload = selected_workload(args)
    flops_one, run, text = oracle_sample(workload, args.reference_rows)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = flops_one * args.steps / el / 1e12
    cfg = describe(workload)
    cfg["sample"] = text
    line = {
        "impl": "reference",
        "metric": "block-scaled GEMM TFLOPS (2MNK/t) and % of GB300 dense FP8/FP4 tensor peak",
        "value": round(value, 6), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded draws with the pages' shapes and distributions)",
        "config": cfg,
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": text + " per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def selected_workload(args) -> W.Workload:
    if args.problem:
        m, n, k = (int(v) for v in args.problem.split(","))
        return W.Workload(f"block_scaled_mm m={m} n={n} k={k}", W.GROUPED_SWEEP.seed, (W.Grouped(m, n, k),))
    return WORKLOADS_BY_KEY[args.workload or "sweep"]


WORKLOADS_BY_KEY = {"sweep": W.GROUPED_SWEEP, "small": W.GROUPED_SMALL, "int8": W.INT8_4096,
                    "mxfp8": W.MXFP8_BATCHED, "nvfp4": W.NVFP4_SQUARE, "mxfp4": W.MXFP4_SQUARE,
                    "backward": W.BACKWARD}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS_BY_KEY), default=None,
                    help="one configuration alone (default: the sweep headline with every other "
                         "configuration as a sub-record)")
    ap.add_argument("--headline-only", action="store_true", help="the default run without the sub-records")
    ap.add_argument("--sub-cpu-seconds", type=float, default=4.0,
                    help="CPU oracle seconds for each sub-record's baseline")
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
