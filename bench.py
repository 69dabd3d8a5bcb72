"""Benchmark: Float8 linear forward + backward (dynamic tensorwise scaling).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

One step = every linear of the workload through the whole path: amax(X),
cast_transpose(X), amax(W), cast_transpose(W), GEMM Y = XW^T, amax(dY),
cast_transpose(dY), GEMM dX = dY W, GEMM dW = dY^T X (the last two in one
launch where the tile schedule gains, as f8_linear_bwd runs them).  The
metric is GEMM work (6 M N K flops per linear) over the whole step's time,
in TFLOP/s.

Inputs are seeded synthetic bf16 tensors (float8_mixed_precision_gb300.workloads),
resident in HBM before timing.  By default the step (every launch of every
linear, made through f8_linear_fwd / f8_linear_bwd) is captured once as a
CUDA graph and replayed each timed step (--graph 0: called each step).  A
step's inputs (0.5 GB for the attention workload, 1.6 GB for the block)
exceed the 129 MB L2, so no L2 flush is inserted between steps.

The JSON line carries, besides the contract keys:
  roofline      the GEMM kernel: GEMM flops of the step over the summed
                duration of its GEMM launches (CUDA events on the launch
                stream, averaged over a timed run of the same steps), against
                the measured bf16 peak x 2 (the FP8 : BF16 dense ratio);
  kernels       the same breakdown for the quantisation of a tensor
                (amax launch + cast_transpose launch, as the linear runs
                them; algorithmic bytes 2 B/elem read + 2 x 1 B/elem
                written, the cast's re-read of the tensor not counted), its
                DRAM bytes from an ncu capture, and bounds on what it adds
                to the replayed step (in_step); the GEMMs' time replayed
                alone as a graph (graph_ms_per_step);
  kernels_isolated  each kernel alone on the workload's tensors, L2 flushed;
  e2e           the same metric through the public API with pinned host
                buffers: inputs copied in and Y, dX, dW copied out every step;
  cpu_baseline  the CPU oracle on a bounded sample of the same workload.
With torchrun (N > 1) every rank runs an independent replica on its own GPU
(no collective on the data path); value = all ranks' work / max time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 linear fwd+bwd TFLOP/s at Llama-3.1-8B shapes; % of GB300 FP8 peak"
UNIT = "TFLOP/s"
FP8_NOMINAL_TFLOPS = 4500.0
FP8_PER_BF16 = 2.0          # nominal dense FP8 : BF16 tensor throughput
HBM_NOMINAL_GBS = 8000.0
REF_BUDGET_S = 60.0   # timed seconds of the CPU reference arm

# DRAM bytes (read + write) of all GEMM launches, and of all quantisation
# launches (amax and cast), of one step of the default workload (the
# Llama-3.1-8B block with its shared-input groups), from one ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum with --cache-control none
# (1 pass, so each launch runs once and finds L2 as the step left it; a
# launch's writes include earlier launches' lines that L2 evicts then, and
# the two figures sum to the step's DRAM traffic); valid for the sources
# whose hash is given, reported as null once they change.
GEMM_TRAFFIC = {"workload": 5, "groups": 1, "bytes_per_step": 5402765568,
                "sources_sha256_16": "892b84bb809b734d"}
QUANT_TRAFFIC = {"workload": 5, "groups": 1, "bytes_per_step": 3936916480,
                 "sources_sha256_16": "37d659e29b0fe522"}


def sources_hash(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "float8_mixed_precision_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_sources_hash() -> str:
    return sources_hash(("f8_gemm.cu", "f8_ptx.cuh", "f8_sched.h"))


def quant_sources_hash() -> str:
    return sources_hash(("f8_cast.cu", "f8_ptx.cuh"))


def captured_traffic(rec: dict, args, current_hash: str):
    """The captured DRAM bytes per step, if they were taken on this workload
    and on the sources as they are now; else None."""
    if (rec["bytes_per_step"] is None or args.config != rec["workload"]
            or int(args.groups) != rec["groups"] or args.fuse_shared_inputs
            or args.swiglu_input != "given" or current_hash != rec["sources_sha256_16"]):
        return None
    return rec["bytes_per_step"]


# ------------------------------------------------------------------ helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
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
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 100 ms"}


class NvmlClockSampler:
    """SM clock, clock-event reasons and power read through NVML (libnvidia-ml,
    read-only queries) every `period_s` by a thread while the timed region
    runs: a region of tens of milliseconds gets tens of samples, where
    nvidia-smi's 100 ms loop gives one.  Falls back to ClockSampler if NVML
    cannot be loaded or the device cannot be found."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        self.gpu = gpu_index
        self.period = period_s
        self.samples = []
        self.fallback = None
        self.nvml = None
        self.max_mhz = None

    def _open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        found = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.gpu).uuid)
            name = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            found = lib.nvmlDeviceGetHandleByUUID(name.encode(), ctypes.byref(h)) == 0
        except Exception:
            found = False
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(self.gpu, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self.nvml, self.h, self.ct = lib, h, ctypes

    def _run(self):
        ct, lib, h = self.ct, self.nvml, self.h
        clk, rs, mw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0:
                r = rs.value if self.reason_fn(h, ct.byref(rs)) == 0 else 0
                p = mw.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else None
                self.samples.append((float(clk.value), int(r), p))
            self.stop.wait(self.period)

    def __enter__(self):
        try:
            self._open()
        except Exception:
            self.fallback = ClockSampler(self.gpu).__enter__()
            return self
        self.stop = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.fallback is not None:
            return self.fallback.__exit__(*exc)
        self.stop.set()
        self.thread.join(timeout=2)

    def summary(self):
        if self.fallback is not None:
            return self.fallback.summary()
        sm = [c for c, _, _ in self.samples]
        reasons = set()
        for _, r, _ in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        power = [p for _, _, p in self.samples if p is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(sm) if sm else None, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None,
                "source": f"NVML, every {self.period * 1e3:g} ms"}


def gpu_local_cpus(gpu_index: int):
    """The CPUs NVML names as closest to the GPU (nvmlDeviceGetCpuAffinity, a
    read-only query), or None.  The e2e leg runs on them so that its pinned
    host buffers are allocated, and first touched, on the GPU's NUMA node."""
    try:
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(gpu_index).uuid)
            name = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = lib.nvmlDeviceGetHandleByUUID(name.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(gpu_index, ctypes.byref(h)) != 0:
            return None
        words = 16
        mask = (ctypes.c_ulong * words)()
        if lib.nvmlDeviceGetCpuAffinity(h, words, mask) != 0:
            return None
        bits = ctypes.sizeof(ctypes.c_ulong) * 8
        cpus = {w * bits + b for w in range(words) for b in range(bits) if (mask[w] >> b) & 1}
        return cpus & os.sched_getaffinity(0) or None
    except Exception:
        return None


def fp8_peak_for(seconds: float, peaks: dict) -> tuple[float, str]:
    """The FP8 dense peak a rate measured over a region of `seconds` is held
    to: the measured bf16 GEMM peak x 2 (the FP8 : BF16 dense ratio), burst
    for a region shorter than a second, sustained (the power-capped
    seconds-long loop) otherwise."""
    if seconds < 1.0:
        return peaks["bf16_tflops"] * FP8_PER_BF16, "burst"
    return peaks["bf16_tflops_sustained"] * FP8_PER_BF16, "sustained"


# ------------------------------------------------------------------ our arm
class Linear8:
    """Device buffers of one linear: inputs, outputs, saved tensors, workspace."""


    def __init__(self, f8, lin, inputs, device, dy_fmt=0, swiglu=None, ab=None):
        import torch
        self.lin = lin
        self.dy_fmt = dy_fmt
        # swiglu: None (X given), "materialized" (h = silu(a) * b by torch each
        # step, then the linear) or "fused" (f8_linear_fwd_swiglu on a, b)
        self.swiglu = swiglu
        if swiglu is not None:
            self.a, self.b = ab[0].to(device), ab[1].to(device)
            self.h = torch.empty_like(self.a)
        self.x = inputs["x"].to(device)
        self.w = inputs["w"].to(device)
        self.dy = inputs["dy"].to(device)
        M, N, K = lin.M, lin.N, lin.K
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=device)
        self.saved = f8.LinearSaved.empty(M, N, K, device)
        self.ws = f8.workspace(M, N, K, device)
        # the decomposed path (same kernels, launched one by one) for per-kernel timing
        self.xq = torch.empty((M, K), dtype=torch.uint8, device=device)
        self.wq = torch.empty((N, K), dtype=torch.uint8, device=device)
        self.dyq = torch.empty((M, N), dtype=torch.uint8, device=device)
        self.dyt = torch.empty((N, M), dtype=torch.uint8, device=device)
        self.dys = torch.empty(2, dtype=torch.float32, device=device)
        self.qws = torch.empty(max(f8.f8_quantize_workspace_bytes(),
                                   f8.f8_quantize_multi_workspace_bytes()),
                               dtype=torch.uint8, device=device)

    @property
    def lins(self):
        return [self.lin]

    def inputs(self):
        """Device tensors a step reads (filled from the host in the e2e run)."""
        return [self.x, self.w, self.dy]

    def outputs(self):
        """Device tensors a step writes (read back in the e2e run)."""
        return [self.y, self.dx, self.dw]

    def iso_items(self):
        """(linear, X, W, dY) of each linear, for the isolated kernel timings."""
        return [(self.lin, self.x, self.w, self.dy)]

    def twin(self, f8, device):
        """A second layer of the same shapes with buffers of its own (the
        e2e leg alternates two, so host copies of one step overlap the
        compute of the other)."""
        ab = (self.a.clone(), self.b.clone()) if self.swiglu is not None else None
        return Linear8(f8, self.lin, {"x": self.x.clone(), "w": self.w.clone(),
                                      "dy": self.dy.clone()}, device, self.dy_fmt, self.swiglu, ab)

    def step(self, f8):
        if self.swiglu == "fused":
            f8.f8_linear_fwd_swiglu(self.a, self.b, self.w, self.y, self.saved, self.ws, h=self.h)
        else:
            if self.swiglu == "materialized":
                import torch
                torch.mul(torch.nn.functional.silu(self.a), self.b, out=self.x)
            f8.f8_linear_fwd(self.x, self.w, self.y, self.saved, self.ws)
        f8.f8_linear_bwd(self.dy, self.saved, dx=self.dx, dw=self.dw, ws=self.ws, dy_fmt=self.dy_fmt)

    def step_timed(self, f8, ev):
        """The same launches as step(), one C call per kernel, bracketed by events."""
        s = self.saved
        M, N, K = self.lin.M, self.lin.N, self.lin.K
        if self.swiglu == "fused":
            ev("quantize", 4 * self.x.numel(),
               lambda: f8.f8_quantize_swiglu(self.a, self.b, self.h, s.amax_x, s.scale_x, self.xq, s.x_t,
                                             self.qws))
        else:
            if self.swiglu == "materialized":
                import torch
                ev("swiglu (torch)", 6 * self.x.numel(),
                   lambda: torch.mul(torch.nn.functional.silu(self.a), self.b, out=self.x))
            # X and W as f8_linear_fwd quantises them: one launch pair when
            # their bf16 bytes fit its L2 budget, else one pair each
            ev("quantize", 4 * (self.x.numel() + self.w.numel()),
               lambda: f8.f8_quantize_multi([self.x, self.w], ws=self.qws, outs=[
                   (self.xq, s.x_t, s.scale_x, s.amax_x), (self.wq, s.w_t, s.scale_w, s.amax_w)]))
        if self.swiglu == "fused":
            ev("quantize", 4 * self.w.numel(),
               lambda: f8.f8_quantize(self.w, s.amax_w, s.scale_w, self.wq, s.w_t, self.qws))
        ev("gemm", 2 * M * N * K, lambda: f8.f8_gemm(self.xq, self.wq, s.scale_x, s.scale_w, self.y))
        self.bwd_timed(f8, ev)

    def bwd_timed(self, f8, ev):
        s = self.saved
        M, N, K = self.lin.M, self.lin.N, self.lin.K
        ev("quantize", 4 * self.dy.numel(),
           lambda: f8.f8_quantize(self.dy, self.dys[0], self.dys[1], self.dyq, self.dyt, self.qws,
                                  fmt=self.dy_fmt))
        # dgrad and wgrad in one launch, as f8_linear_bwd runs them
        ev("gemm", 4 * M * N * K, lambda: f8.f8_gemm_grouped(
            [(self.dyq, s.w_t, self.dys[1], s.scale_w, self.dx, self.dy_fmt),
             (self.dyt, s.x_t, self.dys[1], s.scale_x, self.dw, self.dy_fmt)]))


class GroupLinear8:
    """Linears that read one input X (q, k, v; w1, w3) as one group:
    f8_linear_fwd_group quantises X once and every W_i with its own scale
    (two launches for all of them), then runs the members' GEMMs under the
    grouped-launch planner; f8_linear_bwd_group quantises every dY_i (two
    launches) and runs the members' dgrad and wgrad GEMMs the same way.
    Every output is bit-identical to f8_linear_fwd / f8_linear_bwd on that
    member with the same X."""

    def __init__(self, f8, lins, x, ws, dys, device, dy_fmt=0):
        import torch
        self.members = lins
        self.dy_fmt = dy_fmt
        M, K = lins[0].M, lins[0].K
        self.M, self.K = M, K
        self.Ns = [l.N for l in lins]
        self.lin = type(lins[0])("+".join(l.name for l in lins), M, K, sum(self.Ns))
        self.x = x.to(device)
        self.w = [w.to(device) for w in ws]
        self.dy = [d.to(device) for d in dys]
        self.y = [torch.empty((M, N), dtype=torch.bfloat16, device=device) for N in self.Ns]
        self.dx = [torch.empty((M, K), dtype=torch.bfloat16, device=device) for _ in self.Ns]
        self.dw = [torch.empty((N, K), dtype=torch.bfloat16, device=device) for N in self.Ns]
        self.saved = f8.group_saved(M, K, self.Ns, device)
        self.ws = f8.group_workspace(M, K, self.Ns, device)
        # the decomposed path (same kernels, one C call per phase) for per-phase timing
        self.xq = torch.empty((M, K), dtype=torch.uint8, device=device)
        self.wq = [torch.empty((N, K), dtype=torch.uint8, device=device) for N in self.Ns]
        self.dyq = [torch.empty((M, N), dtype=torch.uint8, device=device) for N in self.Ns]
        self.dyt = [torch.empty((N, M), dtype=torch.uint8, device=device) for N in self.Ns]
        self.dys = [torch.empty(2, dtype=torch.float32, device=device) for _ in self.Ns]
        self.qws = torch.empty(f8.f8_quantize_multi_workspace_bytes(), dtype=torch.uint8,
                               device=device)

    @property
    def lins(self):
        return list(self.members)

    def inputs(self):
        return [self.x] + self.w + self.dy

    def outputs(self):
        return self.y + self.dx + self.dw

    def iso_items(self):
        return [(l, self.x, w, dy) for l, w, dy in zip(self.members, self.w, self.dy)]

    def twin(self, f8, device):
        return GroupLinear8(f8, self.members, self.x.clone(), [w.clone() for w in self.w],
                            [d.clone() for d in self.dy], device, self.dy_fmt)

    def step(self, f8):
        f8.f8_linear_fwd_group(self.x, self.w, ys=self.y, saved=self.saved, ws=self.ws)
        f8.f8_linear_bwd_group(self.dy, self.saved, self.K, dxs=self.dx, dws=self.dw, ws=self.ws,
                               fmt=self.dy_fmt)

    def step_timed(self, f8, ev):
        s = self.saved
        xs = s[0].x_scalars
        outs = [(self.xq, s[0].x_t, xs[1], xs[0])] + [
            (wq, si.w_t, si.scalars[3], si.scalars[2]) for wq, si in zip(self.wq, s)]
        ev("quantize", 4 * (self.x.numel() + sum(w.numel() for w in self.w)),
           lambda: f8.f8_quantize_multi([self.x] + self.w, outs=outs, ws=self.qws))
        (_, fwd_flops, fwd), (_, bwd_flops, bwd) = self.gemm_calls(f8)
        ev("gemm", fwd_flops, fwd)
        douts = [(q, t, d[1], d[0]) for q, t, d in zip(self.dyq, self.dyt, self.dys)]
        ev("quantize", 4 * sum(d.numel() for d in self.dy),
           lambda: f8.f8_quantize_multi(self.dy, fmt=self.dy_fmt, outs=douts, ws=self.qws))
        ev("gemm", bwd_flops, bwd)

    def gemm_calls(self, f8):
        """The group's forward GEMMs and its backward GEMMs, each as the
        one f8_gemm_grouped call the group makes (the planner decides the
        launches): [(label, flops, call), ...] on the decomposed path's
        quantised operands."""
        s = self.saved
        M, K = self.M, self.K
        xs = s[0].x_scalars
        fwd = [(self.xq, wq, xs[1], si.scalars[3], y) for wq, si, y in zip(self.wq, s, self.y)]
        bwd = []
        for i in range(len(self.Ns)):
            bwd.append((self.dyq[i], s[i].w_t, self.dys[i][1], s[i].scalars[3], self.dx[i],
                        self.dy_fmt))
            bwd.append((self.dyt[i], s[i].x_t, self.dys[i][1], xs[1], self.dw[i], self.dy_fmt))
        ns = "+".join(str(N) for N in self.Ns)
        return [(f"{self.lin.name} fwd M={M} K={K} N={ns}", sum(2 * M * N * K for N in self.Ns),
                 lambda: f8.f8_gemm_grouped(fwd)),
                (f"{self.lin.name} dgrad+wgrad M={M} K={K} N={ns}",
                 sum(4 * M * N * K for N in self.Ns), lambda: f8.f8_gemm_grouped(bwd))]


class FfnIn8(Linear8):
    """The group {w1, w3} of a SwiGLU FFN (W13 interleaved by 128 rows) with
    the SwiGLU epilogue: f8_linear_fwd_w13_swiglu writes AB (into y), h and
    q(h), q(h)^T and h's amax and scale for the W2Q8 that follows, then the
    group's backward."""

    def __init__(self, f8, lin, inputs, device, dy_fmt=0, chain=False):
        import torch
        super().__init__(f8, lin, inputs, device, dy_fmt)
        M, F = lin.M, lin.N // 2
        self.h = torch.empty((M, F), dtype=torch.bfloat16, device=device)
        self.h_q = torch.empty((M, F), dtype=torch.uint8, device=device)
        self.next = None  # the W2Q8 whose saved tensors receive q(h)^T and h's scalars
        # chain: the group's dY is not given but formed from dh by the SwiGLU
        # backward, which the W2Q8 runs after its own backward
        self.chain = chain
        if chain:
            self.dy = torch.empty_like(self.y)  # d(AB), written each step

    def step(self, f8):
        s2 = self.next.saved
        f8.f8_linear_fwd_w13_swiglu(self.x, self.w, self.y, self.h, self.saved, s2.scalars[0:1],
                                    s2.scalars[1:2], self.h_q, s2.x_t, self.ws)
        if not self.chain:
            f8.f8_linear_bwd(self.dy, self.saved, dx=self.dx, dw=self.dw, ws=self.ws,
                             dy_fmt=self.dy_fmt)

    def bwd_from_dh(self, f8, dh):
        f8.f8_linear_bwd_w13_swiglu(dh, self.y, self.saved, dab=self.dy, dx=self.dx, dw=self.dw,
                                    ws=self.ws, dy_fmt=self.dy_fmt)

    def bwd_from_dh_timed(self, f8, ev, dh):
        s = self.saved
        M, N, K = self.lin.M, self.lin.N, self.lin.K
        # reads dh, a, b (6 B per element of h) and writes d(AB) (4 B), then the cast
        ev("quantize", 10 * dh.numel() + 4 * self.dy.numel(),
           lambda: f8.f8_quantize_swiglu_bwd(dh, self.y, self.dy, self.dys[0], self.dys[1], self.dyq,
                                             self.dyt, self.qws, fmt=self.dy_fmt))
        # dgrad and wgrad in one launch, as f8_linear_bwd runs them
        ev("gemm", 4 * M * N * K, lambda: f8.f8_gemm_grouped(
            [(self.dyq, s.w_t, self.dys[1], s.scale_w, self.dx, self.dy_fmt),
             (self.dyt, s.x_t, self.dys[1], s.scale_x, self.dw, self.dy_fmt)]))

    def step_timed(self, f8, ev):
        s, s2 = self.saved, self.next.saved
        M, N, K = self.lin.M, self.lin.N, self.lin.K
        ev("quantize", 4 * self.x.numel(),
           lambda: f8.f8_quantize(self.x, s.amax_x, s.scale_x, self.xq, s.x_t, self.qws))
        ev("quantize", 4 * self.w.numel(),
           lambda: f8.f8_quantize(self.w, s.amax_w, s.scale_w, self.wq, s.w_t, self.qws))
        ev("gemm", 2 * M * N * K,
           lambda: f8.f8_gemm_w13_swiglu(self.xq, self.wq, s.scale_x, s.scale_w, self.y, self.h,
                                         s2.scalars[0:1]))
        ev("quantize", 4 * self.h.numel(),
           lambda: f8.f8_cast_transpose(self.h, s2.scalars[0:1], s2.scalars[1:2], self.h_q, s2.x_t))
        if not self.chain:
            self.bwd_timed(f8, ev)


class W2Q8(Linear8):
    """The w2 linear fed by the q(h) that its FfnIn8 produced: W2 quantised
    (f8_quantize), the GEMM on q(h) (f8_gemm), then the linear's backward."""

    def __init__(self, f8, lin, inputs, device, dy_fmt, src: FfnIn8):
        super().__init__(f8, lin, inputs, device, dy_fmt)
        self.src = src
        src.next = self

    def step(self, f8):
        s = self.saved
        f8.f8_quantize(self.w, s.amax_w, s.scale_w, self.wq, s.w_t, self.qws)
        f8.f8_gemm(self.src.h_q, self.wq, s.scale_x, s.scale_w, self.y)
        f8.f8_linear_bwd(self.dy, self.saved, dx=self.dx, dw=self.dw, ws=self.ws, dy_fmt=self.dy_fmt)
        if self.src.chain:
            self.src.bwd_from_dh(f8, self.dx)  # dX of w2 is dh

    def step_timed(self, f8, ev):
        s = self.saved
        M, N, K = self.lin.M, self.lin.N, self.lin.K
        ev("quantize", 4 * self.w.numel(),
           lambda: f8.f8_quantize(self.w, s.amax_w, s.scale_w, self.wq, s.w_t, self.qws))
        ev("gemm", 2 * M * N * K,
           lambda: f8.f8_gemm(self.src.h_q, self.wq, s.scale_x, s.scale_w, self.y))
        self.bwd_timed(f8, ev)
        if self.src.chain:
            self.src.bwd_from_dh_timed(f8, ev, self.dx)


def describe_workload(wl, args):
    """The workload's name and the linears one step runs (as build_layers
    makes them), from the arguments alone: both arms print it as `config`."""
    name, lins = wl.workload(args.config)
    if args.swiglu_input in ("epilogue", "chain"):
        if args.config not in wl.SHARED_INPUT_GROUPS:
            raise SystemExit("--swiglu-input epilogue needs a workload with a SwiGLU FFN (3, 4, 5)")
        chain = args.swiglu_input == "chain"
        return (name + " (shared inputs fused; w2 input silu(a) * b from the w1+w3 GEMM epilogue"
                + ("; dY of w1+w3 from the SwiGLU backward of dX of w2)" if chain else ")"),
                [g for g, _ in wl.fused_groups(args.config)])
    if args.fuse_shared_inputs:
        groups = [g for g, _ in wl.fused_groups(args.config)]
        name += " (shared inputs fused: " + ", ".join(g.name for g in groups) + ")"
        lins = groups
    elif use_groups(wl, args):
        name += (" (linears that share X as groups: " +
                 ", ".join("+".join(g) for g in wl.SHARED_INPUT_GROUPS[args.config] if len(g) > 1) +
                 "; X quantised once, one scale per tensor)")
    if args.swiglu_input != "given" and any(l.x_kind == "swiglu" for l in lins):
        name += f" (w2 input: silu(a) * b, {args.swiglu_input})"
    return name, lins


def use_groups(wl, args) -> bool:
    """Whether the step runs the linears that share X as groups
    (f8_linear_fwd_group / f8_linear_bwd_group)."""
    return (args.groups and args.config in wl.SHARED_INPUT_GROUPS and not args.fuse_shared_inputs
            and args.swiglu_input == "given")


def config_dict(wl, args, world):
    name, lins = describe_workload(wl, args)
    return {"workload": name,
            "linears": [f"{l.name} M={l.M} K={l.K} N={l.N}" for l in lins],
            "flops_per_step": sum(l.flops for l in lins),
            "parallelism": "replicas" if world > 1 else "single-gpu",
            "l2": "no flush: a step's inputs exceed L2",
            "launch": "one captured CUDA graph per step" if args.graph else "call by call"}


def build_layers(f8, wl, args, device, dy_fmt):
    """The workload's linears as layer objects, and the workload's name."""
    name, _ = describe_workload(wl, args)
    lins = wl.workload(args.config)[1]
    if args.swiglu_input in ("epilogue", "chain"):
        chain = args.swiglu_input == "chain"
        if args.config not in wl.SHARED_INPUT_GROUPS:
            raise SystemExit("--swiglu-input epilogue needs a workload with a SwiGLU FFN (3, 4, 5)")
        layers, ffn = [], None
        for g, idx in wl.fused_groups(args.config):
            if g.name == "w1+w3":
                ffn = FfnIn8(f8, g, wl.w13_group_inputs(args.config, idx), device, dy_fmt, chain)
                layers.append(ffn)
            elif g.name == "w2" and ffn is not None:
                layers.append(W2Q8(f8, g, wl.fused_group_inputs(args.config, idx), device, dy_fmt,
                                   ffn))
            else:
                layers.append(Linear8(f8, g, wl.fused_group_inputs(args.config, idx), device,
                                      dy_fmt))
        if ffn is None:
            raise SystemExit("--swiglu-input epilogue needs a workload with a SwiGLU FFN (3, 4, 5)")
        return name, layers
    if use_groups(wl, args):
        by_name = {l.name: i for i, l in enumerate(lins)}
        layers = []
        for names in wl.SHARED_INPUT_GROUPS[args.config]:
            idx = [by_name[n] for n in names]
            if len(idx) == 1:
                layers.append(Linear8(f8, lins[idx[0]], wl.linear_inputs(args.config, idx[0]),
                                      device, dy_fmt))
                continue
            ins = [wl.linear_inputs(args.config, i) for i in idx]
            layers.append(GroupLinear8(f8, [lins[i] for i in idx], ins[0]["x"],
                                       [d["w"] for d in ins], [d["dy"] for d in ins], device,
                                       dy_fmt))
        return name, layers
    if args.fuse_shared_inputs:
        layers = []
        for g, idx in wl.fused_groups(args.config):
            sw = (args.swiglu_input if g.x_kind == "swiglu" and args.swiglu_input != "given"
                  else None)
            layers.append(Linear8(f8, g, wl.fused_group_inputs(args.config, idx), device, dy_fmt,
                                  sw, wl.swiglu_ab(args.config, idx[0]) if sw else None))
    else:
        layers = []
        for i, lin in enumerate(lins):
            sw = args.swiglu_input if (lin.x_kind == "swiglu" and args.swiglu_input != "given") else None
            layers.append(Linear8(f8, lin, wl.linear_inputs(args.config, i), device, dy_fmt, sw,
                                  wl.swiglu_ab(args.config, i) if sw else None))
    return name, layers


def run_ours(args, world, rank, local):
    import torch

    import float8_mixed_precision_gb300 as f8
    from float8_mixed_precision_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    f8.lib()
    dy_fmt = f8.F8_E5M2 if args.dy_format == "e5m2" else f8.F8_E4M3
    name, layers = build_layers(f8, wl, args, device, dy_fmt)
    lins = [l for L in layers for l in L.lins]
    flops_step = sum(l.flops for l in lins)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- warm-up, then the timed region (library calls f8_linear_fwd/bwd)
    for _ in range(args.warmup):
        n0 = f8.f8_kernel_launches()
        for L in layers:
            L.step(f8)
        launches_per_step = f8.f8_kernel_launches() - n0  # counted by libf8 itself
    graph = None
    if args.graph:
        # one whole step (every launch of every linear) captured once and replayed
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for L in layers:
                    L.step(f8)
        stream.wait_stream(cap)
        for _ in range(2):
            graph.replay()
    st = f8.f8_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {f8.f8_status_string(st)}")
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    busy_t0 = time.perf_counter()
    with NvmlClockSampler(local) as clocks:
        t0.record(stream)
        for _ in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                for L in layers:
                    L.step(f8)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1)
    st = f8.f8_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status after the timed region: {f8.f8_status_string(st)}")
    ms_max = max_over_ranks(ms, world, device)
    total_flops = sum_over_ranks(flops_step * args.steps, world, device)
    value = total_flops / (ms_max * 1e-3) / 1e12

    # ---- per-kernel breakdown: the same kernels, each bracketed by events
    nsteps_k = max(1, min(args.steps, 100))
    rec = []

    def ev(kind, work, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        rec.append((kind, work, a, b))

    for _ in range(2):
        for L in layers:
            L.step_timed(f8, lambda k, w, fn: fn())
    torch.cuda.synchronize()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for _ in range(nsteps_k):
        for L in layers:
            L.step_timed(f8, ev)
    k1.record(stream)
    torch.cuda.synchronize()
    breakdown_ms = k0.elapsed_time(k1) / nsteps_k
    per = {}
    for kind, work, a, b in rec:
        d = per.setdefault(kind, {"launches": 0, "ms": 0.0, "work": 0.0})
        d["launches"] += 1
        d["ms"] += a.elapsed_time(b)
        d["work"] += work
    tot_ms = sum(d["ms"] for d in per.values())

    # ---- the step's GEMM launches alone, captured as a graph of their own
    # (on the operands the replay above quantised): the replayed step's time
    # minus theirs is what the quantisation adds to the replayed step, with
    # programmatic launch overlapping neighbours as in the step itself
    gemm_graph_ms = None
    if args.graph:
        torch.cuda.synchronize()
        gg = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gg, stream=cap):
                for L in layers:
                    L.step_timed(f8, lambda k, w, fn: fn() if k == "gemm" else None)
        stream.wait_stream(cap)
        for _ in range(2):
            gg.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(nsteps_k):
            gg.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gemm_graph_ms = g0.elapsed_time(g1) / nsteps_k
        del gg
    peaks = load_peaks()
    # the GPU has been busy from the start of the timed region to here: the
    # burst peak applies to a region under a second, the sustained one beyond
    busy_s = time.perf_counter() - busy_t0
    fp8_peak, regime = fp8_peak_for(busy_s, peaks)
    kernels = {}
    for kind, d in per.items():
        rate = d["work"] / (d["ms"] * 1e-3)
        e = {"launches_per_step": d["launches"] // nsteps_k, "ms_per_step": d["ms"] / nsteps_k,
             "share": d["ms"] / tot_ms}
        if kind == "swiglu (torch)":
            e.update({"gbs": rate / 1e9})
        elif kind == "gemm":
            e.update({"tflops": rate / 1e12, "frac_of_fp8_measured": rate / 1e12 / fp8_peak,
                      "fp8_peak_regime": regime,
                      "frac_of_fp8_nominal": rate / 1e12 / FP8_NOMINAL_TFLOPS})
        else:
            e.update({"gbs": rate / 1e9, "frac_of_hbm_measured": rate / 1e9 / peaks["hbm_gbs"],
                      "frac_of_hbm_nominal": rate / 1e9 / HBM_NOMINAL_GBS})
            if kind == "quantize":
                # DRAM bytes the quantisation launches move (ncu), against the
                # algorithmic 4 B per element (2 read + 2 written)
                qt = captured_traffic(QUANT_TRAFFIC, args, quant_sources_hash())
                e.update({"algorithmic_bytes_per_step": d["work"] / nsteps_k,
                          "dram_bytes_per_step": qt,
                          "dram_over_algorithmic": (qt / (d["work"] / nsteps_k)) if qt else None,
                          "dram_gbs": (qt / (d["ms"] / nsteps_k * 1e-3) / 1e9) if qt else None,
                          # the same time against the bytes DRAM really moved, and the
                          # best frac_of_hbm_measured those bytes allow (every byte at
                          # the copy rate, no launch costs): the two-pass ceiling
                          "dram_frac_of_hbm_measured": ((qt / (d["ms"] / nsteps_k * 1e-3) / 1e9)
                                                        / peaks["hbm_gbs"]) if qt else None,
                          "two_pass_ceiling_frac": ((d["work"] / nsteps_k) / qt) if qt else None})
        if gemm_graph_ms is not None and kind == "gemm":
            e.update({"graph_ms_per_step": gemm_graph_ms,
                      "graph_tflops": d["work"] / nsteps_k / (gemm_graph_ms * 1e-3) / 1e12})
        if gemm_graph_ms is not None and kind == "quantize":
            # what the quantisation adds to the replayed step, bounded from
            # below two ways: the step minus the event-timed GEMM calls, and
            # the step minus the GEMM launches replayed alone as one graph.
            # Both GEMM figures exceed the GEMMs' share of the replayed step
            # (the calls pay their launch ramp without programmatic overlap;
            # back to back, the GEMMs run hotter and slower), so both
            # differences are lower bounds on the quantisation's time and
            # their fractions upper bounds on its rate.  frac_of_hbm_measured
            # above, from per-call events that include each call's launch,
            # is a lower bound.
            step_ms = ms_max / args.steps
            alg = d["work"] / nsteps_k
            g_ev = per["gemm"]["ms"] / nsteps_k

            def frac(q_ms):
                return alg / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"] if q_ms > 0 else None
            e["in_step"] = {
                "step_minus_gemm_calls": {"ms_per_step": step_ms - g_ev,
                                          "frac_of_hbm_measured": frac(step_ms - g_ev)},
                "step_minus_gemm_graph": {"ms_per_step": step_ms - gemm_graph_ms,
                                          "frac_of_hbm_measured": frac(step_ms - gemm_graph_ms)}}
        kernels[kind] = e
    g = per["gemm"]
    achieved = g["work"] / (g["ms"] * 1e-3) / 1e12
    roofline = {"kernel": "gemm_kernel (tcgen05 kind::f8f6f4)", "bound": "tensor",
                "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak,
                "peak_regime": regime,
                "peak_note": (f"{peaks['source']} bf16 {regime} "
                              f"{peaks['bf16_tflops' if regime == 'burst' else 'bf16_tflops_sustained']}"
                              f" x {FP8_PER_BF16} (FP8:BF16 dense); {regime} because the GPU was busy "
                              f"{busy_s:.2f} s from the start of the timed region to the end of the "
                              f"per-kernel replay (burst below 1 s)"),
                "frac_of_burst": achieved / (peaks["bf16_tflops"] * FP8_PER_BF16),
                "frac_of_sustained": achieved / (peaks["bf16_tflops_sustained"] * FP8_PER_BF16),
                "frac_of_nominal_4500": achieved / FP8_NOMINAL_TFLOPS,
                "traffic": captured_traffic(GEMM_TRAFFIC, args, gemm_sources_hash()),
                "traffic_unit": "bytes per step (all GEMM launches of the step, like achieved)",
                # E4M3 operands read once + bf16 outputs written once, 3 GEMMs per linear
                "algorithmic_bytes_per_step": sum(4 * (l.M * l.K + l.N * l.K + l.M * l.N)
                                                  for l in lins)}

    # the chained FFN's w2 reads a device-made input: no isolated or host-fed runs
    chained = args.swiglu_input in ("epilogue", "chain")
    iso = kernel_bench(f8, layers, device, stream) if args.kernel_bench and not chained else None

    # ---- end to end: pinned host buffers in, results out, every step
    e2e = None
    if args.e2e_steps > 0 and not chained:
        e2e = run_e2e(f8, layers, args, device, stream, flops_step, world)

    return {"value": value, "ms_per_step": ms_max / args.steps, "name": name, "lins": lins,
            "clocks": clocks.summary(), "kernels": kernels, "roofline": roofline,
            "breakdown_ms_per_step": breakdown_ms, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "isolated": iso}


def kernel_bench(f8, layers, device, stream, iters=50):
    """Each kernel timed alone on the workload's tensors: 10 warm-up
    launches, then the median of `iters`, with L2 flushed before every
    launch (a 1 GiB fill, then a 256 MB read so that the L2 holds clean
    lines and the timed kernel pays no write-back for the flush) and CUDA
    events around the launch only.
    amax: 2 B/elem read; cast_transpose: 2 B/elem read + 2 x 1 B/elem
    written; GEMM: 2 M N K flops.  f8_amax includes its 4-byte memset."""
    import torch
    flush = torch.empty(1024 * 1024 * 1024, dtype=torch.uint8, device=device)
    clean = torch.ones(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    peaks = load_peaks()
    fp8_burst = peaks["bf16_tflops"] * FP8_PER_BF16

    def timed(fn):
        ts = []
        for _ in range(10):  # warm-up launches
            fn()
        for _ in range(iters):
            flush.fill_(1)                # evicts everything from L2 ...
            clean.max()                   # ... then fills it with clean lines
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    out = []
    seen = set()
    for L in layers:
        for lin, x, w, dy in L.iso_items():
            M, N, K = lin.M, lin.N, lin.K
            dy_fmt = L.dy_fmt
            amx = {}
            ops = {}
            for name, t in (("x", x), ("w", w), ("dy", dy)):
                amx[name] = torch.empty((), dtype=torch.float32, device=device)
                q = torch.empty(t.shape, dtype=torch.uint8, device=device)
                qt = torch.empty((t.shape[1], t.shape[0]), dtype=torch.uint8, device=device)
                sc = torch.empty((), dtype=torch.float32, device=device)
                ws = torch.empty(f8.f8_quantize_workspace_bytes(), dtype=torch.uint8, device=device)
                fmt = dy_fmt if name == "dy" else 0
                f8.f8_quantize(t, amx[name], sc, q, qt, ws, fmt=fmt)   # operands for the GEMMs
                ops[name] = (q, qt, sc)
                key = ("mem", tuple(t.shape))
                if key in seen:
                    continue
                seen.add(key)
                a1 = amx[name]
                ms = timed(lambda: f8.f8_amax(t, a1))
                out.append({"kernel": "amax", "tensor": f"{lin.name}.{name} {list(t.shape)}",
                            "us": ms * 1e3, "gbs": 2 * t.numel() / ms / 1e6,
                            "frac_of_hbm_measured": 2 * t.numel() / ms / 1e6 / peaks["hbm_gbs"],
                            "frac_of_hbm_nominal": 2 * t.numel() / ms / 1e6 / HBM_NOMINAL_GBS})
                ms = timed(lambda: f8.f8_cast_transpose(t, a1, sc, q, qt))
                out.append({"kernel": "cast_transpose", "tensor": f"{lin.name}.{name} {list(t.shape)}",
                            "us": ms * 1e3, "gbs": 4 * t.numel() / ms / 1e6,
                            "frac_of_hbm_measured": 4 * t.numel() / ms / 1e6 / peaks["hbm_gbs"],
                            "frac_of_hbm_nominal": 4 * t.numel() / ms / 1e6 / HBM_NOMINAL_GBS})
                ms = timed(lambda: f8.f8_quantize(t, a1, sc, q, qt, ws, fmt=fmt))
                out.append({"kernel": "quantize (amax + cast_transpose launches)",
                            "tensor": f"{lin.name}.{name} {list(t.shape)}", "us": ms * 1e3,
                            "gbs": 4 * t.numel() / ms / 1e6,
                            "frac_of_hbm_measured": 4 * t.numel() / ms / 1e6 / peaks["hbm_gbs"],
                            "frac_of_hbm_nominal": 4 * t.numel() / ms / 1e6 / HBM_NOMINAL_GBS,
                            "note": "4 B/elem counted (2 read + 2 written); the cast's re-read is not"})
            (xq, xt, sx), (wq, wt, sw), (dyq, dyt, sdy) = ops["x"], ops["w"], ops["dy"]
            for gname, (a, b, sa, sb, mm, nn, kk) in (
                    ("fwd", (xq, wq, sx, sw, M, N, K)),
                    ("dgrad", (dyq, wt, sdy, sw, M, K, N)),
                    ("wgrad", (dyt, xt, sdy, sx, N, K, M))):
                key = ("gemm", mm, nn, kk)
                if key in seen:
                    continue
                seen.add(key)
                fa = dy_fmt if gname != "fwd" else 0
                c = torch.empty((mm, nn), dtype=torch.bfloat16, device=device)
                ms = timed(lambda: f8.f8_gemm(a, b, sa, sb, c, fmt_a=fa))
                tf = 2 * mm * nn * kk / ms / 1e9
                out.append({"kernel": "gemm", "shape": f"{lin.name}.{gname} M={mm} N={nn} K={kk}",
                            "us": ms * 1e3, "tflops": tf, "frac_of_fp8_measured_burst": tf / fp8_burst,
                            "frac_of_fp8_nominal": tf / FP8_NOMINAL_TFLOPS})
                del c
            del ops
        if isinstance(L, GroupLinear8):
            # the members' GEMMs as the step launches them: the skinny wk, wv
            # (or w1, w3) problems share launches with the others
            for label, flops, fn in L.gemm_calls(f8):
                ms = timed(fn)
                tf = flops / ms / 1e9
                out.append({"kernel": "gemm (the group's grouped call)", "shape": label,
                            "us": ms * 1e3, "tflops": tf,
                            "frac_of_fp8_measured_burst": tf / fp8_burst,
                            "frac_of_fp8_nominal": tf / FP8_NOMINAL_TFLOPS})
    del flush, clean
    return out


def run_e2e(f8, layers, args, device, stream, flops_step, world):
    """The whole step from pinned host buffers and back, through the public
    API.  Three streams form a pipeline (host-to-device copies, compute,
    device-to-host copies) over two sets of device buffers used by
    alternate steps: the copies into one set overlap the compute and the
    read-back of the other, and events order each buffer's reuse (a set's
    inputs are overwritten only after its previous compute has read them,
    its compute starts only after its previous outputs have been read
    back)."""
    import torch
    # run on the GPU's NUMA-local CPUs while the pinned buffers are made and
    # used (first touch places them on that node); restored at the end
    old_aff = os.sched_getaffinity(0)
    local = gpu_local_cpus(device.index if device.index is not None else 0)
    if local:
        os.sched_setaffinity(0, local)
    sets = [layers, [L.twin(f8, device) for L in layers]]
    host = []
    h2d = d2h = 0
    for L in layers:
        hin = [t.cpu().pin_memory() for t in L.inputs()]
        hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in L.outputs()]
        host.append((hin, hout))
        h2d += sum(t.numel() * t.element_size() for t in hin)
        d2h += sum(t.numel() * t.element_size() for t in hout)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    n = len(layers)
    ev_in = [[torch.cuda.Event() for _ in range(n)] for _ in sets]
    ev_comp = [[torch.cuda.Event() for _ in range(n)] for _ in sets]
    ev_out = [[torch.cuda.Event() for _ in range(n)] for _ in sets]
    used = [[False] * n for _ in sets]
    count = [0]

    def step():
        k = count[0] % 2
        count[0] += 1
        for i, (L, (hin, hout)) in enumerate(zip(sets[k], host)):
            with torch.cuda.stream(s_in):
                if used[k][i]:
                    s_in.wait_event(ev_comp[k][i])   # this set's last compute has read its inputs
                for d, h in zip(L.inputs(), hin):
                    d.copy_(h, non_blocking=True)
                ev_in[k][i].record(s_in)
            stream.wait_event(ev_in[k][i])
            if used[k][i]:
                stream.wait_event(ev_out[k][i])      # this set's last outputs have been read back
            L.step(f8)
            ev_comp[k][i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[k][i])
                for h, d in zip(hout, L.outputs()):
                    h.copy_(d, non_blocking=True)
                ev_out[k][i].record(s_out)
            used[k][i] = True

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    # several timed windows of e2e_steps steps each; the median window is
    # the figure (the host link of these boxes stalls now and then for
    # 0.1-0.2 s, which would otherwise decide a single short window)
    window_ms = []
    for _ in range(max(1, args.e2e_windows)):
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for _ in range(args.e2e_steps):
            step()
        s_out.wait_stream(stream)
        t1.record(s_out)
        torch.cuda.synchronize()
        window_ms.append(max_over_ranks(t0.elapsed_time(t1), world, device))
    ms = sorted(window_ms)[len(window_ms) // 2]
    total = sum_over_ranks(flops_step * args.e2e_steps, world, device)
    # the results really came back: spot-check one output of the last step
    last = sets[(count[0] - 1) % 2]
    ok = torch.equal(host[-1][1][-1][:4].to(device), last[-1].outputs()[-1][:4])
    del sets[1]
    link = host_link_gbs(device, s_in, s_out)
    moved = (h2d + d2h) * args.e2e_steps / (ms * 1e-3) / 1e9
    os.sched_setaffinity(0, old_aff)
    return {"value": total / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "ms_per_step": ms / args.e2e_steps,
            "windows": len(window_ms), "statistic": "median window",
            "window_values": [total / (w * 1e-3) / 1e12 for w in window_ms],
            "pipelined": "3 streams (h2d, compute, d2h), two buffer sets on alternate steps",
            "readback_check": bool(ok), "host_bytes_gbs": moved,
            "host_link_gbs_measured": link, "frac_of_host_link": moved / link if link else None,
            "host_cpus": (f"{len(local)} GPU-local CPUs (NVML affinity)" if local
                          else "no NVML affinity: unbound")}


def host_link_gbs(device, s_in, s_out, nbytes=512 << 20, reps=6):
    """Pinned host<->device bandwidth of this machine with both directions busy
    at once (as in the e2e step): bytes moved both ways / time, after one
    untimed round that touches every page."""
    import torch
    hs = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    hd = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    ds = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dd = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def both():
        with torch.cuda.stream(s_in):
            ds.copy_(hs, non_blocking=True)
        with torch.cuda.stream(s_out):
            hd.copy_(dd, non_blocking=True)

    both()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(reps):
        both()
    torch.cuda.synchronize()
    sec = time.perf_counter() - t0
    return 2 * nbytes * reps / sec / 1e9


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(config: int, lin_index: int, rows: int):
    """The oracle on a bounded sample of one linear: amax, scale and cast of X,
    W and dY in full, then ``rows`` output rows of each of the three GEMMs.
    Returns (GEMM flops of the sampled rows, seconds, seconds per phase)."""
    import numpy as np

    import oracle
    from float8_mixed_precision_gb300 import workloads as wl

    lin = wl.workload(config)[1][lin_index]
    d = wl.linear_inputs(config, lin_index)
    xb, wb, dyb = wl.bits(d["x"]), wl.bits(d["w"]), wl.bits(d["dy"])
    rng = np.random.default_rng(lin_index)
    M, N, K = lin.M, lin.N, lin.K
    r_m = np.sort(rng.choice(M, size=min(rows, M), replace=False))
    r_n = np.sort(rng.choice(N, size=min(rows, N), replace=False))
    t0 = time.perf_counter()
    amaxes = [oracle.amax(b)[0] for b in (xb, wb, dyb)]
    t1 = time.perf_counter()
    scales = [oracle.scale(a) for a in amaxes]
    (xq, xt), (wq, wt), (dyq, dyt) = [oracle.cast_transpose(b, sc)
                                      for b, sc in zip((xb, wb, dyb), scales)]
    t2 = time.perf_counter()
    sx, sw, sdy = scales
    oracle.gemm_rows(xq, wq, sx, sw, r_m)          # Y rows
    oracle.gemm_rows(dyq, wt, sdy, sw, r_m)        # dX rows
    oracle.gemm_rows(dyt, xt, sdy, sx, r_n)        # dW rows
    t3 = time.perf_counter()
    flops = 2 * (len(r_m) * N * K + len(r_m) * K * N + len(r_n) * K * M)
    return flops, t3 - t0, {"amax": t1 - t0, "scale+cast_transpose": t2 - t1, "gemm": t3 - t2}


def cpu_baseline(config: int, rows: int):
    import oracle
    from float8_mixed_precision_gb300 import workloads as wl
    flops, sec, phases = oracle_sample(config, 0, rows)
    lins = wl.workload(config)[1]
    lin = lins[0]
    rm, rn = min(rows, lin.M), min(rows, lin.N)
    # the whole step on the same cores, from the measured rates: the GEMMs at
    # the sample's GEMM rate, the quantisation at its measured bf16 bytes/s
    gemm_rate = flops / phases["gemm"] if flops > 0 and phases["gemm"] > 0 else None
    q_s = phases["amax"] + phases["scale+cast_transpose"]
    q_rate = 2 * (lin.M * lin.K + lin.N * lin.K + lin.M * lin.N) / q_s if q_s > 0 else None
    step_s = (sum(l.flops / gemm_rate + 2 * (l.M * l.K + l.N * l.K + l.M * l.N) / q_rate
                  for l in lins) if gemm_rate and q_rate else None)
    return {"value": flops / sec / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": sec,
            "seconds_by_phase": phases,
            "gemm_gflops": gemm_rate / 1e9 if gemm_rate else None,
            "extrapolated_step_seconds": step_s,
            "extrapolated_note": ("extrapolated: the whole workload step on these cores at the "
                                  "sample's measured GEMM and quantisation rates"),
            "sample": (f"linear {lin.name} (M={lin.M}, K={lin.K}, N={lin.N}): amax, scale and "
                       f"cast of X, W, dY in full, then {rm} of {lin.M} output rows of Y and of "
                       f"dX and {rn} of {lin.N} rows of dW; value = GEMM flops of those rows / "
                       f"wall time")}


class OracleSampler:
    """Bounded samples of the oracle's work on one workload, for the CPU
    reference arm.  Inputs and their full quantisation are built once per
    linear (untimed); a timed sample is the oracle's amax + scale + cast of
    the first `frac` of the rows of X, W and dY plus `rows` sampled output
    rows of each of the three GEMMs, so the sample keeps the step's mix of
    quantisation and GEMM work."""

    def __init__(self, config: int):
        from float8_mixed_precision_gb300 import workloads as wl
        self.config = config
        self.lins = wl.workload(config)[1]
        self.cache = {}

    def _prep(self, i):
        if i not in self.cache:
            import oracle
            from float8_mixed_precision_gb300 import workloads as wl
            d = wl.linear_inputs(self.config, i)
            b = {k: wl.bits(v) for k, v in d.items()}
            self.cache[i] = (b, {k: oracle.quantize(v) for k, v in b.items()})
        return self.cache[i]

    def sample(self, i: int, rows: int):
        import numpy as np

        import oracle
        b, q = self._prep(i)
        lin = self.lins[i]
        M, N, K = lin.M, lin.N, lin.K
        rng = np.random.default_rng(rows + 7 * i)
        r_m = np.sort(rng.choice(M, size=min(rows, M), replace=False))
        r_n = np.sort(rng.choice(N, size=min(rows, N), replace=False))
        frac = len(r_m) / M
        t = time.perf_counter()
        for key in ("x", "w", "dy"):
            part = b[key][: max(1, int(round(frac * b[key].shape[0])))]
            oracle.quantize(part)
        qx, qw, qdy = q["x"], q["w"], q["dy"]
        oracle.gemm_rows(qx["q"], qw["q"], qx["scale"], qw["scale"], r_m)
        oracle.gemm_rows(qdy["q"], qw["qt"], qdy["scale"], qw["scale"], r_m)
        oracle.gemm_rows(qdy["qt"], qx["qt"], qdy["scale"], qx["scale"], r_n)
        sec = time.perf_counter() - t
        flops = 2 * (len(r_m) * N * K + len(r_m) * K * N + len(r_n) * K * M)
        return flops, sec


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle, as it stands, timed on the host cores.
    The per-step sample is sized so that the timed steps take about
    REF_BUDGET_S seconds whatever --steps is."""
    import oracle
    from float8_mixed_precision_gb300 import workloads as wl
    name, lins = wl.workload(args.config)
    if rank != 0:
        return 0
    oracle.build()
    sampler = OracleSampler(args.config)
    for i in range(len(lins)):
        sampler._prep(i)
    # calibrate: seconds per sampled row on this host
    f0, t0 = sampler.sample(0, 16)
    per_row = t0 / 16
    target = max(0.02, min(5.0, REF_BUDGET_S / max(1, args.steps)))
    rows = int(max(1, min(lins[0].M, target / per_row)))
    for i in range(args.warmup):
        sampler.sample(i % len(lins), max(1, rows // 4))
    flops = sec = 0.0
    for i in range(args.steps):
        f, s_ = sampler.sample(i % len(lins), rows)
        flops += f
        sec += s_
    value = flops / sec / 1e12
    sample = (f"per step one linear (rotating over {', '.join(l.name for l in lins)}): amax, scale "
              f"and cast of the first {rows}/{lins[0].M} of the rows of X, W, dY and {rows} sampled "
              f"output rows of each of Y, dX, dW; value = GEMM flops of the sampled rows / time")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "impl": "reference",
            "config": config_dict(wl, args, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5],
                    help="workload (default 5: the full Llama-3.1-8B block, all seven linears)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20, help="steps per timed e2e window")
    ap.add_argument("--e2e-windows", type=int, default=5,
                    help="timed e2e windows; the median window is reported")
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--ref-rows", type=int, default=128)
    ap.add_argument("--graph", type=int, default=1,
                    help="replay the step as one captured CUDA graph (1) or launch it call by call (0)")
    ap.add_argument("--groups", type=int, default=1,
                    help="run the linears that share X (q, k, v; w1, w3) as groups: X quantised "
                         "once, one scale per tensor, GEMMs in shared launches (1, default) or "
                         "every linear alone (0)")
    ap.add_argument("--fuse-shared-inputs", action="store_true",
                    help="merge the linears that read one input (q/k/v, w1/w3) into one linear "
                         "with the concatenated weight and a tensorwise scale over it")
    ap.add_argument("--swiglu-input", default="given",
                    choices=["given", "materialized", "fused", "epilogue", "chain"],
                    help="for linears fed by silu(a) * b: the bf16 product given (default), "
                         "formed by torch each step, produced from given a, b with its amax "
                         "(f8_linear_fwd_swiglu), or formed in the epilogue of the w1+w3 "
                         "group's GEMM and fed to w2 (implies --fuse-shared-inputs); chain: "
                         "epilogue, and the group's dY formed from dX of w2 by the SwiGLU "
                         "backward (only dY of w2 given)")
    ap.add_argument("--dy-format", default="e4m3", choices=["e4m3", "e5m2"],
                    help="FP8 format of dY in the backward pass (X and W stay E4M3)")
    ap.add_argument("--kernel-bench", type=int, default=1,
                    help="also time each kernel alone with L2 flushed (1) or not (0)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cpu = None
    if rank == 0:
        # the CPU oracle runs first, before any GPU work in this process
        cpu = cpu_baseline(args.config, args.cpu_rows) if world == 1 else None
    r = run_ours(args, world, rank, local)
    if rank == 0:
        from float8_mixed_precision_gb300 import workloads as wl
        line = {
            "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if args.dy_format == "e4m3" else "e4m3 (X, W) / e5m2 (dY)",
            "data": "synthetic (seeded; workloads.py)",
            "config": config_dict(wl, args, world),
            "pct_of_fp8_peak_nominal": 100 * r["value"] / FP8_NOMINAL_TFLOPS,
            "roofline": r["roofline"], "kernels": r["kernels"],
            "breakdown_ms_per_step": r["breakdown_ms_per_step"],
            "clocks": r["clocks"], "gpu_launches": r["gpu_launches"],
            "kernels_isolated": r["isolated"],
            "e2e": r["e2e"], "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
