"""Benchmark of the fine-grained FP8 hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

One step is one pass of the whole path over one batch: quantize the bf16
activations per 1x128 tile, quantize the bf16 weights per 128x128 block
(weights change every training step, so they are re-quantized each step),
and run the block-scaled FP8 GEMM with FP32 promotion. The default workload
is the dense 7168-square layer (A [8192, 7168] with outlier channels,
B [7168, 7168]); --config 4 times the grouped MoE GEMM path instead
(32768 routed rows, 256 experts of [2048, 7168]); --config 2 / 6 time the MLA
down-projections as two GEMMs / as one GEMM on the stacked Wq||Wkv; --config 7
runs the MoE step as quantize-the-tokens-then-dispatch-in-FP8.

The printed JSON line reports whole-step TFLOP/s (2*M*N*K per step over the
step time), the per-kernel times (CUDA events on the launching stream), the
GEMM's roofline against the FP8 tensor peak, an end-to-end figure through
the public API with pinned host buffers, the CPU oracle timed on a bounded
sample of the same workload, and the SM clocks sampled during the timed
region. Multi-GPU (torchrun): every rank runs its own copy of the workload
(weak scaling, no collective on the data path); the time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("block-scaled FP8 GEMM TFLOPS (% of B300 FP8 peak); quantize GB/s (% HBM)")
FP8_OVER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor throughput (4.5 : 2.25 PFLOP/s)
BURST_REGION_S = 1.0  # a timed region shorter than this runs at burst clocks unless capped
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def code_hash(path: str) -> str:
    """First 16 hex digits of the sha256 of a C/C++/CUDA source with its
    comments and all whitespace removed, so that editing a comment does not
    unlink a profile taken on the same code."""
    with open(path) as fh:
        src = fh.read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":  # string or character literal, kept whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    code = "".join("".join(out).split())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def profiled_traffic(profile: str, source: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    recorded in profiles/<profile> by an ncu capture, or None when the
    kernel code changed since (its recorded code hash differs)."""
    try:
        with open(os.path.join(ROOT, "profiles", profile)) as fh:
            text = fh.read()
        cur = code_hash(os.path.join(ROOT, "fp8_fine_grained_25_b300", "csrc", source))
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(re.escape(source) + r" ([0-9a-f]{16})", text)
    if m and h and h.group(1) == cur:
        return int(m.group(1))
    return None


# ------------------------------------------------------------------ clocks
_REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
            ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))


class ClockSampler:
    """SM clock and clock-event reasons of one GPU, polled from a host thread
    every `period_s` (in-process NVML; nvidia-smi at 100 ms if NVML is not
    available), each sample stamped with the host clock so that a summary
    can be taken over any window (the timed region, a probe)."""

    def __init__(self, device: torch.device, period_s: float = 0.001):
        self.device = device
        self.period_s = period_s
        self.samples = []          # (host seconds, sm MHz, max sm MHz, reasons bitmask)
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    @staticmethod
    def _nvml(device):
        """(read_fn, max_mhz) for the GPU behind `device`, through the NVML
        library that ships with the driver (libnvidia-ml, via ctypes)."""
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        p = torch.cuda.get_device_properties(device)
        bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device.index or 0), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for the device")
        NVML_CLOCK_SM = 1
        mhz, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        if nv.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) != 0:
            raise OSError("nvmlDeviceGetMaxClockInfo failed")

        def read():
            if nv.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mhz)) != 0:
                return None
            if reasons(h, ctypes.byref(bits)) != 0:
                bits.value = 0
            return float(mhz.value), int(bits.value)
        return read, float(mx.value)

    def __enter__(self):
        try:
            read, max_mhz = self._nvml(self.device)

            def poll():
                while not self._stop.is_set():
                    t = time.perf_counter()
                    r = read()
                    if r is not None:
                        self.samples.append((t, r[0], max_mhz, r[1]))
                    self._stop.wait(self.period_s)
            self.source = f"NVML (libnvidia-ml) every {self.period_s * 1e3:.0f} ms"
            self._thread = threading.Thread(target=poll, daemon=True)
            self._thread.start()
        except (OSError, AttributeError) as ex:
            self.nvml_error = str(ex)
            self._start_smi()
        return self

    def _start_smi(self):
        fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active")
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0), f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.source = "nvidia-smi every 100 ms"

        def read():
            for line in self._proc.stdout:
                parts = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((time.perf_counter(), float(parts[0]), float(parts[1]),
                                         int(parts[2], 16)))
                except (ValueError, IndexError):
                    continue
        self._thread = threading.Thread(target=read, daemon=True)
        self._thread.start()

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, t0: float = float("-inf"), t1: float = float("inf")):
        """Median SM clock, the maximum clock and the union of the clock-event
        reasons that were active, over the samples taken in [t0, t1]."""
        sel = [x for x in list(self.samples) if t0 <= x[0] <= t1]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        bits = 0
        for x in sel:
            bits |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
                "reasons": [n for n, b in _REASONS if bits & b], "samples": len(sel),
                "source": self.source}


# ------------------------------------------------------- FP8 tensor ceiling
NOMINAL_FP8_TFLOPS = 4500.0  # B300 dense FP8 datasheet figure (context)


def fp8_ceiling(device, clocks: ClockSampler, seconds: float = 2.0):
    """The FP8 dense tensor ceiling measured on this GPU with cuBLAS
    (torch._scaled_mm, per-tensor scales, E4M3 x E4M3 -> bf16, 8192^3).
    Reported beside the GEMM only; nothing on the measured path uses it.
    burst: the best mean over five runs of 20 back-to-back launches (the
    length of a short timed region); sustained: back to back for `seconds`
    (long enough for the power limit to act)."""
    n = 8192
    g = torch.Generator(device=device).manual_seed(12345)
    a = torch.randn(n, n, generator=g, device=device).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, generator=g, device=device).to(torch.float8_e4m3fn)
    one = torch.ones((), device=device)
    f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    flop = 2.0 * n ** 3

    def run(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            f()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    try:
        for _ in range(5):
            f()
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        best = min(run(20) for _ in range(5))
        h1 = time.perf_counter()
        reps = max(20, int(seconds / best))
        tsus = run(reps)
        h2 = time.perf_counter()
    except RuntimeError as ex:  # no FP8 GEMM in this torch/cuBLAS build
        return {"unavailable": str(ex).splitlines()[0][:200]}
    finally:
        del a, b
    return {"how": "cuBLAS via torch._scaled_mm, per-tensor scales, E4M3 x E4M3 -> bf16, 8192^3",
            "burst_tflops": flop / best / 1e12, "burst_clocks": clocks.summary(h0, h1),
            "sustained_tflops": flop / tsus / 1e12, "sustained_s": tsus * reps,
            "sustained_clocks": clocks.summary(h1, h2)}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(seconds: float, dist=None, device=None) -> float:
    """The job time of one timed region: the slowest rank's time (every
    rank runs its own replica; no data moves between ranks)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_step: float, steps: int, seconds: float) -> float:
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's time."""
    return world * flops_per_step * steps / seconds / 1e12


# ---------------------------------------------------------------- workloads
def make_workload(config: int, device, experts: int = 0):
    """The workload of `config`; for the MoE configs (4, 7) `experts` > 0
    keeps `experts` of the 256 routed experts and the same tokens per expert
    (T = 4096 * experts / 256), a smaller case of the same layer."""
    from fp8_fine_grained_25_b300 import workloads
    if experts and config in (4, 7):
        return workloads.WORKLOADS[config](seed=0, device=device, E=experts,
                                           T=max(workloads.TOP_K, 4096 * experts // workloads.N_ROUTED))
    return workloads.WORKLOADS[config](seed=0, device=device)


def step_flops(w) -> float:
    if w.X is not None:  # backward of a dense layer: the dX and dW GEMMs
        T, N = w.A.shape
        return 2.0 * 2.0 * T * N * w.X.shape[1]
    M, K = w.A.shape
    if w.offsets is not None:
        N = w.weights["W"].shape[1]
    else:
        N = next(iter(w.weights.values())).shape[0] if len(w.weights) == 1 else None
    if N is None:  # several weights against the same A (MLA: Wq and Wkv)
        return float(sum(2.0 * M * W.shape[0] * K for W in w.weights.values()))
    return 2.0 * M * N * K


def args_dispatch(w) -> bool:
    return w.index is not None and "dispatch" in w.name


class Path:
    """The forward hot path on one device: buffers allocated once, one call
    per step. inputs() / outputs() name the step's bf16 inputs and its
    outputs; step() takes replacements for either (the end-to-end run
    passes freshly copied inputs and its own output buffers)."""

    def __init__(self, w, device):
        from fp8_fine_grained_25_b300 import fp8q
        self.fp8q = fp8q
        self.w = w
        A = w.A
        M, K = A.shape
        self.ue8m0 = w.scales == "ue8m0"
        sdt = torch.uint8 if self.ue8m0 else torch.float32  # UE8M0 scale bytes or fp32 scales
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=device)
        self.sa = torch.empty((M, -(-K // 128)), dtype=sdt, device=device)
        self.bufs = {}
        for name, W in w.weights.items():
            qb = torch.empty(W.shape, dtype=torch.uint8, device=device)
            if W.dim() == 3:
                sb = torch.empty((W.shape[0], W.shape[1] // 128, -(-K // 128)), dtype=torch.float32,
                                 device=device)
                C = torch.empty((M, W.shape[1]), dtype=torch.bfloat16, device=device)
            else:
                sb = torch.empty((-(-W.shape[0] // 128), -(-K // 128)), dtype=sdt, device=device)
                C = torch.empty((M, W.shape[0]), dtype=torch.bfloat16, device=device)
            self.bufs[name] = (qb, sb, C)
        # split-K workspace of each dense FP32-scale GEMM whose shape splits
        # (the MLA down-projections); none for shapes that do not
        self.ws = {}
        if w.offsets is None and not self.ue8m0:
            for name, W in w.weights.items():
                n = fp8q.fp8_block_gemm_workspace_size(M, W.shape[0], K)
                if n > 0:
                    self.ws[name] = torch.empty(n, dtype=torch.uint8, device=device)
        self.launches_per_step = 1 + 2 * len(w.weights)
        # FP8 dispatch: quantize the T tokens, then gather rows into expert order
        self.dispatch = args_dispatch(w)
        if self.dispatch:
            T = w.tokens.shape[0]
            self.qx = torch.empty((T, K), dtype=torch.uint8, device=device)
            self.sx = torch.empty((T, -(-K // 128)), dtype=torch.float32, device=device)
            self.launches_per_step += 1
        self.flops = step_flops(w)
        self.names = (["quant_act"] + [f"quant_weight[{n}]" for n in w.weights]
                      + [f"gemm[{n}]" for n in w.weights])
        self.gemm_names = [f"gemm[{n}]" for n in w.weights]
        self.dominant = self.gemm_names  # the roofline kernel(s)
        self.dominant_flops = self.flops
        self.describe = describe(w)

    def inputs(self):
        return step_inputs(self.w)

    def outputs(self):
        return {n: self.bufs[n][2] for n in self.w.weights}

    def step(self, inp=None, outs=None, events=None, stream=None, only=None):
        """One pass of the path on `stream` (default: the current one);
        `only` names the one kernel of `names` to launch by itself."""
        f = self.fp8q
        inp = self.inputs() if inp is None else inp
        A = inp["A"]
        rec = (lambda i: events[i].record(stream)) if events is not None else (lambda i: None)
        run = lambda name: only is None or only == name
        rec(0)
        if not run("quant_act"):
            pass
        elif self.dispatch:
            f.fp8q_quant_act(A, self.qx, self.sx, stream=stream)
            f.fp8q_gather_rows(self.qx, self.sx, self.w.index, self.qa, self.sa, stream=stream)
        elif self.ue8m0:
            f.fp8q_quant_act_ue8m0(A, self.qa, self.sa, stream=stream)
        else:
            f.fp8q_quant_act(A, self.qa, self.sa, stream=stream)
        rec(1)
        i = 2
        for name in self.w.weights:
            qb, sb, _ = self.bufs[name]
            if not run(f"quant_weight[{name}]"):
                pass
            elif self.ue8m0:
                f.fp8q_quant_weight_ue8m0(inp[name], qb, sb, stream=stream)
            else:
                f.fp8q_quant_weight(inp[name], qb, sb, stream=stream)
            rec(i)
            i += 1
        for name in self.w.weights:
            qb, sb, C = self.bufs[name]
            if outs is not None:
                C = outs[name]
            if not run(f"gemm[{name}]"):
                pass
            elif self.w.offsets is not None:
                f.fp8_grouped_gemm(self.qa, self.sa, qb, sb, self.w.offsets, C, stream=stream)
            elif self.ue8m0:
                f.fp8_block_gemm_ue8m0(self.qa, self.sa, qb, sb, C, stream=stream)
            elif name in self.ws:
                f.fp8_block_gemm_ws(self.qa, self.sa, qb, sb, C, workspace=self.ws[name], stream=stream)
            else:
                f.fp8_block_gemm(self.qa, self.sa, qb, sb, C, stream=stream)
            rec(i)
            i += 1

    def kernels(self, per):
        """Per-kernel time and throughput from the per-launch seconds `per`."""
        w = self.w
        M, K = w.A.shape
        kern = {}
        if self.dispatch:
            T = w.tokens.shape[0]
            qbytes = 3 * T * K + 4 * T * -(-K // 128) + 2 * (M * K + 4 * M * -(-K // 128))
            kern["quant_act+dispatch"] = {"ms": per["quant_act"] * 1e3,
                                          "GB/s": qbytes / per["quant_act"] / 1e9}
        else:
            kern["quant_act"] = {"ms": per["quant_act"] * 1e3,
                                 "GB/s": (3 * M * K + 4 * M * -(-K // 128)) / per["quant_act"] / 1e9}
        for n, W in w.weights.items():
            e = W.numel()
            blocks = e // W.shape[-1] // 128 * -(-W.shape[-1] // 128)
            tq = per[f"quant_weight[{n}]"]
            kern[f"quant_weight[{n}]"] = {"ms": tq * 1e3, "GB/s": (3 * e + 4 * blocks) / tq / 1e9}
            N = W.shape[-2]
            tg = per[f"gemm[{n}]"]
            kern[f"gemm[{n}]"] = {"ms": tg * 1e3, "TFLOP/s": 2.0 * M * N * K / tg / 1e12}
        return kern


class BackwardPath:
    """The backward pass of a dense FP8 layer y = x W^T on one device:
        quant_act(dY) -> qdy                      (1x128 tiles)
        quant_weight_t(W) -> qt(W)                (128x128 blocks, transposed codes)
        dX = fp8_block_gemm(qdy, qt(W))           (input gradient, [T, K])
        quant_act_t(dY), quant_act_t(X)           (128x1 tiles along tokens)
        dW = fp8_wgrad_gemm(dY^T codes, X^T codes) (weight gradient, [N, K])"""

    def __init__(self, w, device):
        from fp8_fine_grained_25_b300 import fp8q
        self.fp8q = fp8q
        self.w = w
        dY, X, W = w.A, w.X, w.weights["W"]
        T, N = dY.shape
        K = X.shape[1]
        e = lambda *shape, dt=torch.uint8: torch.empty(shape, dtype=dt, device=device)
        self.ue8m0 = w.scales == "ue8m0"
        sdt = torch.uint8 if self.ue8m0 else torch.float32  # UE8M0 bytes or fp32 scales
        self.qdy, self.sdy = e(T, N), e(T, -(-N // 128), dt=sdt)
        self.qwt, self.swt = e(K, N), e(-(-K // 128), -(-N // 128), dt=sdt)
        self.qdyt, self.sdyt = e(N, T), e(N, -(-T // 128), dt=sdt)
        self.qxt, self.sxt = e(K, T), e(K, -(-T // 128), dt=sdt)
        self.dX = e(T, K, dt=torch.bfloat16)
        self.dW = e(N, K, dt=torch.bfloat16)
        self.T, self.N, self.K = T, N, K
        self.launches_per_step = 6
        self.dispatch = False
        self.flops = 2.0 * (2.0 * T * N * K)
        self.names = ["quant_act[dY]", "quant_weight_t[W]", "gemm[dX]", "quant_act_t[dY]",
                      "quant_act_t[X]", "gemm[dW]"]
        self.gemm_names = ["gemm[dX]", "gemm[dW]"]
        self.dominant = ["gemm[dW]"]  # the largest share of the step
        self.dominant_flops = 2.0 * T * N * K
        self.describe = describe(w)

    def inputs(self):
        return step_inputs(self.w)

    def outputs(self):
        return {"dX": self.dX, "dW": self.dW}

    def step(self, inp=None, outs=None, events=None, stream=None, only=None):
        f = self.fp8q
        inp = self.inputs() if inp is None else inp
        outs = self.outputs() if outs is None else outs
        rec = (lambda i: events[i].record(stream)) if events is not None else (lambda i: None)
        run = lambda name: only is None or only == name
        rec(0)
        u = self.ue8m0
        if run("quant_act[dY]"):
            (f.fp8q_quant_act_ue8m0 if u else f.fp8q_quant_act)(inp["dY"], self.qdy, self.sdy, stream=stream)
        rec(1)
        if run("quant_weight_t[W]"):
            (f.fp8q_quant_weight_t_ue8m0 if u else f.fp8q_quant_weight_t)(
                inp["W"], qt=self.qwt, st=self.swt, with_forward=False, stream=stream)
        rec(2)
        if run("gemm[dX]"):
            (f.fp8_block_gemm_ue8m0 if u else f.fp8_block_gemm)(self.qdy, self.sdy, self.qwt, self.swt,
                                                                outs["dX"], stream=stream)
        rec(3)
        act_t = f.fp8q_quant_act_t_ue8m0 if u else f.fp8q_quant_act_t
        if run("quant_act_t[dY]"):
            act_t(inp["dY"], self.qdyt, self.sdyt, stream=stream)
        rec(4)
        if run("quant_act_t[X]"):
            act_t(inp["X"], self.qxt, self.sxt, stream=stream)
        rec(5)
        if run("gemm[dW]"):
            (f.fp8_wgrad_gemm_ue8m0 if u else f.fp8_wgrad_gemm)(self.qdyt, self.sdyt, self.qxt, self.sxt,
                                                                outs["dW"], stream=stream)
        rec(6)

    def kernels(self, per):
        T, N, K = self.T, self.N, self.K
        act = lambda rows, cols: 3 * rows * cols + 4 * rows * -(-cols // 128)
        kern = {
            "quant_act[dY]": (per["quant_act[dY]"], act(T, N), None),
            "quant_weight_t[W]": (per["quant_weight_t[W]"],
                                  3 * N * K + 4 * -(-N // 128) * -(-K // 128), None),
            "gemm[dX]": (per["gemm[dX]"], None, 2.0 * T * N * K),
            "quant_act_t[dY]": (per["quant_act_t[dY]"], act(T, N), None),
            "quant_act_t[X]": (per["quant_act_t[X]"], act(T, K), None),
            "gemm[dW]": (per["gemm[dW]"], None, 2.0 * T * N * K),
        }
        out = {}
        for n, (t, nbytes, fl) in kern.items():
            out[n] = {"ms": t * 1e3}
            if nbytes is not None:
                out[n]["GB/s"] = nbytes / t / 1e9
            else:
                out[n]["TFLOP/s"] = fl / t / 1e12
        return out


def step_inputs(w) -> dict:
    """The bf16 tensors one step reads (what the end-to-end run copies in)."""
    if w.X is not None:
        return {"dY": w.A, "X": w.X, "W": w.weights["W"]}
    d = {"A": w.tokens if args_dispatch(w) else w.A}
    d.update(w.weights)
    return d


def describe(w) -> str:
    """The workload and the kernels one step runs (the same for both arms)."""
    if w.X is not None:
        return (w.name + ": quant_act(dY) + quant_weight_t(W) + dX GEMM + "
                "quant_act_t(dY) + quant_act_t(X) + dW GEMM per step")
    return (w.name + ": quant_act(A) + quant_weight(W) + "
            + ("grouped" if w.offsets is not None else "dense")
            + (" hardware-scaled" if w.scales == "ue8m0" else "")
            + " block-scaled GEMM per step")


def run_config(w, world: int) -> dict:
    nbytes = sum(t.numel() * t.element_size() for t in step_inputs(w).values())
    return {"workload": describe(w), "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2 (bf16 inputs {nbytes / 1e6:.0f} MB re-read every step)"}


def make_path(w, device):
    return BackwardPath(w, device) if w.X is not None else Path(w, device)


def time_alone(path, names, device, reps: int = 25):
    """Seconds of each named kernel launched by itself, with a 256 MB read
    just before it so that the L2 holds no dirty lines (inside the step a
    quantizer also writes back the previous kernel's output) and none of its
    input. CUDA event timestamps on the B300 advance in steps of 2.048 us, so
    one launch of ~30 us is timed to +-7 %: the result is the mean of the
    middle 15 of `reps` launches, which averages that out (a median would
    stay on the 2.048 us grid) and drops outliers (a plain mean would not)."""
    clean = torch.ones(256 << 20, dtype=torch.uint8, device=device)
    out = {}
    for n in names:
        for _ in range(3):
            path.step(only=n)
        ts = []
        for _ in range(reps):
            clean.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            path.step(only=n)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        ts.sort()
        out[n] = statistics.fmean(ts[(reps - 15) // 2:(reps - 15) // 2 + 15])
    del clean
    return out


# --------------------------------------------------------------- CPU oracle
def _busy(units: int, threads: int) -> float:
    """Fraction of the oracle's host threads a call over `units` independent
    rows (or row blocks) keeps busy: the oracle splits them over threads."""
    return min(units, threads) / threads


def oracle_sample(w, rows_a: int, w_rows: int, out_rows: int, threads: int):
    """Time the CPU oracle on a bounded sample of one step and extrapolate
    the full step: quant_act on `rows_a` rows of A, quant_weight on the first
    `w_rows` rows of the (first) weight, and the GEMM of `out_rows` rows of A
    against those weight rows. Each part scales by its work ratio and by the
    share of threads the sample kept busy (a sample with fewer rows than
    threads runs on fewer threads than the full step would).
    Returns (seconds for a full step, description)."""
    import numpy as np
    import oracle
    A = w.A
    M, K = A.shape
    Wd = w.weights["W"][0] if w.offsets is not None else next(iter(w.weights.values()))
    N = Wd.shape[0]
    w_rows, out_rows = min(w_rows, N), min(out_rows, rows_a)
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a_s, b_s = bits(A[:rows_a]), bits(Wd[:w_rows])
    pow2 = w.scales == "ue8m0"
    qact = oracle.quant_act_ue8m0 if pow2 else oracle.quant_act
    qweight = oracle.quant_weight_ue8m0 if pow2 else oracle.quant_weight
    gemm = oracle.gemm_ue8m0 if pow2 else oracle.gemm
    t0 = time.perf_counter()
    qa, sa = qact(a_s, threads=threads)
    t1 = time.perf_counter()
    qb, sb = qweight(b_s, threads=threads)
    t2 = time.perf_counter()
    gemm(qa, sa, qb, sb, rows=np.arange(out_rows), threads=threads)
    t3 = time.perf_counter()
    w_elems = sum(W.numel() for W in w.weights.values())
    full = ((t1 - t0) * (M * K) / a_s.size * _busy(rows_a, threads)
            + (t2 - t1) * w_elems / b_s.size * _busy(-(-w_rows // 128), threads)
            + (t3 - t2) * (step_flops(w) / (2.0 * out_rows * w_rows * K)) * _busy(out_rows, threads))
    desc = (f"oracle quant_act on {rows_a}x{K}, quant_weight on {w_rows}x{K} of a [{N}x{K}] weight, "
            f"GEMM on {out_rows} x {w_rows} outputs; sample took {t3 - t0:.2f} s, full step "
            "extrapolated by work, per busy thread")
    return full, desc


def oracle_sample_backward(w, rows: int, cols: int, out_rows: int, w_cols: int, threads: int):
    """The same for the backward step: quant_act on `rows` rows of dY, the
    transposed weight quantization on the first `w_cols` columns of W, the
    dX GEMM on out_rows x w_cols outputs, quant_act_t on `cols` columns of dY
    and of X, and the dW GEMM on out_rows x cols outputs; each part scaled as
    in oracle_sample."""
    import numpy as np
    import oracle
    dY, X, W = w.A, w.X, w.weights["W"]
    T, N = dY.shape
    K = X.shape[1]
    w_cols = min(w_cols, K)
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    dy_rows, dy_cols, x_cols = bits(dY[:rows]), bits(dY[:, :cols]), bits(X[:, :cols])
    w_part = bits(W[:, :w_cols])
    u = w.scales == "ue8m0"
    qact = oracle.quant_act_ue8m0 if u else oracle.quant_act
    qwt = oracle.quant_weight_t_ue8m0 if u else oracle.quant_weight_t
    gemm = oracle.gemm_ue8m0 if u else oracle.gemm
    qact_t = oracle.quant_act_t_ue8m0 if u else oracle.quant_act_t
    wgrad = oracle.wgrad_gemm_ue8m0 if u else oracle.wgrad_gemm
    t = [time.perf_counter()]
    qdy, sdy = qact(dy_rows, threads=threads)
    t.append(time.perf_counter())
    _, _, qwt_, swt_ = qwt(w_part, threads=threads)
    t.append(time.perf_counter())
    gemm(qdy, sdy, qwt_, swt_, rows=np.arange(out_rows), threads=threads)
    t.append(time.perf_counter())
    qdyt, sdyt = qact_t(dy_cols, threads=threads)
    t.append(time.perf_counter())
    qxt, sxt = qact_t(x_cols, threads=threads)
    t.append(time.perf_counter())
    wgrad(qdyt, sdyt, qxt, sxt, rows=np.arange(out_rows), threads=threads)
    t.append(time.perf_counter())
    d = np.diff(t)
    b = lambda units: _busy(units, threads)
    full = (d[0] * T / rows * b(rows) + d[1] * K / w_cols + d[2] * (T * K) / (out_rows * w_cols) * b(out_rows)
            + d[3] * N / cols * b(cols) + d[4] * K / cols * b(cols)
            + d[5] * (N * K) / (out_rows * cols) * b(out_rows))
    desc = (f"oracle quant_act on {rows} rows of dY, quant_weight_t on {w_cols} columns of W, dX "
            f"GEMM on {out_rows} x {w_cols} outputs, quant_act_t on {cols} columns of dY and of X, "
            f"dW GEMM on {out_rows} x {cols} outputs; sample took {t[-1] - t[0]:.2f} s, full step "
            "extrapolated by work, per busy thread")
    return full, desc


# Oracle sample sizes, largest first: (rows of A, weight rows, GEMM rows) for
# a forward step, (rows of dY, columns of dY/X, GEMM rows, columns of W) for a
# backward one. Tier 0 is the cpu_baseline sample (about 10-30 s of oracle
# work on an 8- to 16-core host); the reference arm takes the largest tier
# that lets all of its steps finish within its time budget. Smaller samples
# still extrapolate to a somewhat slower oracle (per-call costs scale up).
SAMPLE_TIERS = [(4096, 1 << 30, 3072), (2048, 1024, 256), (1024, 512, 128), (512, 256, 64),
                (64, 128, 8)]
SAMPLE_TIERS_BACKWARD = [(4096, 2048, 1536, 1 << 30), (2048, 1024, 256, 1024), (1024, 512, 128, 512),
                         (512, 256, 64, 256), (64, 128, 8, 128)]


def sample_oracle(w, tier: int, threads: int):
    """The bounded oracle sample of one step of workload w at a size tier."""
    if w.X is not None:
        rows, cols, out_rows, w_cols = SAMPLE_TIERS_BACKWARD[tier]
        return oracle_sample_backward(w, rows=rows, cols=cols, out_rows=out_rows, w_cols=w_cols,
                                      threads=threads)
    rows_a, w_rows, out_rows = SAMPLE_TIERS[tier]
    return oracle_sample(w, rows_a=rows_a, w_rows=w_rows, out_rows=out_rows, threads=threads)


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on this machine's cores."""
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    w = make_workload(args.config, "cpu", args.experts)
    flops = step_flops(w)
    # the largest sample tier whose first step, repeated for the whole run,
    # fits the budget (tier 0 is the cpu_baseline sample, too large here)
    budget_s = 240.0
    tier = 1
    while True:
        t0 = time.perf_counter()
        sample_oracle(w, tier, threads)
        if (time.perf_counter() - t0) * (args.warmup + args.steps) <= budget_s or tier == len(SAMPLE_TIERS) - 1:
            break
        tier += 1
    times, measured = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        full, desc = sample_oracle(w, tier, threads)
        if i >= args.warmup:
            times.append(full)
            measured.append(time.perf_counter() - t0)
    t = statistics.median(times)
    value = flops / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "extrapolated": True,
            "measured_sample_s_per_step": statistics.median(measured),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64/f32", "data": "synthetic",
            "config": run_config(w, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def choose_fp8_peak(fp8: dict, peaks: dict, peak_kind: str, timed_s: float, clk: dict):
    """The FP8 tensor peak a GEMM timed over `timed_s` seconds with clock
    record `clk` is measured against: the larger of the FP8 ceiling measured
    in this run (`fp8`, from fp8_ceiling) and 2 x the measured bf16 peak,
    in its burst form when the timed region is under BURST_REGION_S and saw
    no power cap, else in its sustained form.
    Returns (peak, burst peak, sustained peak, description)."""
    bf16_burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    bf16_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP8_OVER_BF16
    burst = max(fp8.get("burst_tflops", 0.0), bf16_burst)
    sus = max(fp8.get("sustained_tflops", 0.0), bf16_sus)
    capped = "sw_power_cap" in clk.get("reasons", [])
    use_burst = timed_s < BURST_REGION_S and not capped
    key, other = ("burst_tflops", bf16_burst) if use_burst else ("sustained_tflops", bf16_sus)
    origin = ("measured fp8 (cuBLAS, this run)" if fp8.get(key, 0.0) >= other
              else f"{peak_kind} bf16 x {FP8_OVER_BF16} (nominal FP8:BF16 ratio)")
    desc = (f"{'burst' if use_burst else 'sustained'}: {origin}; the larger of the measured FP8 "
            f"ceiling and 2 x bf16 ({bf16_burst:.1f} burst, {bf16_sus:.1f} sustained); burst is used "
            f"when the timed region is under {BURST_REGION_S:.0f} s and saw no power cap (this one: "
            f"{timed_s:.3f} s, power cap {'seen' if capped else 'not seen'})")
    return (burst if use_burst else sus), burst, sus, desc


# ------------------------------------------------- kernels at other shapes
def _time_mean(fn, reps: int, clean=None) -> float:
    """Seconds per call: the mean of the middle 60 % of `reps` timed calls
    (each after `clean()`, if given, which is not timed)."""
    for _ in range(3):
        fn()
    ts = []
    for _ in range(reps):
        if clean is not None:
            clean()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    ts.sort()
    k = max(1, int(0.6 * reps))
    lo = (reps - k) // 2
    return statistics.fmean(ts[lo:lo + k])


def extra_legs(device, peaks):
    """After the dense step: the activation quantizer on 32768 x 7168 bf16
    (a large-M batch with outlier channels) and the grouped GEMM of the MoE
    layer (4096 tokens, 256 experts of [2048, 7168], top-8), each launched by
    itself. The quantizer runs after a 256 MB read that leaves no input in
    L2; the grouped GEMM streams 3.76 GB of expert weights, far more than L2.
    The grouped GEMM's roofline is max(FLOPs / FP8 peak, bytes / HBM)."""
    from fp8_fine_grained_25_b300 import fp8q, workloads
    out = {}
    clean_buf = torch.ones(256 << 20, dtype=torch.uint8, device=device)
    clean = lambda: clean_buf.sum()
    M, K = 32768, workloads.HIDDEN
    A = workloads.activations_with_outliers(M, K, seed=5001, device=device)
    qa = torch.empty((M, K), dtype=torch.uint8, device=device)
    sa = torch.empty((M, -(-K // 128)), dtype=torch.float32, device=device)
    t = _time_mean(lambda: fp8q.fp8q_quant_act(A, qa, sa), 25, clean)
    nbytes = 3 * M * K + 4 * M * -(-K // 128)
    out[f"quant_act[{M}x{K}]"] = {"ms": t * 1e3, "GB/s": nbytes / t / 1e9,
                                  "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
                                  "timed": "alone, clean L2, mean of the middle 15 of 25"}
    del A, qa, sa, clean_buf

    w = workloads.moe_grouped(seed=0, device=device)
    W = w.weights["W"]
    E, N, K = W.shape
    M = w.A.shape[0]
    qa, sa = fp8q.fp8q_quant_act(w.A)
    qw, sw = fp8q.fp8q_quant_weight(W)
    del W, w.weights["W"]
    C = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    t = _time_mean(lambda: fp8q.fp8_grouped_gemm(qa, sa, qw, sw, w.offsets, C), 20)
    assert fp8q.fp8q_get_device_status() == 0
    fl = 2.0 * M * N * K
    wbytes = E * N * K + 4 * E * (N // 128) * -(-K // 128)
    abytes = M * K + 4 * M * -(-K // 128) + 2 * M * N
    fp8_peak_est = peaks["bf16_tflops"] * FP8_OVER_BF16 * 1e12  # 2 x bf16 burst
    roof_t = max(fl / fp8_peak_est, (wbytes + abytes) / (peaks["hbm_gbs"] * 1e9))
    out[f"grouped_gemm[MoE T=4096 E={E} top8 {N}x{K}]"] = {
        "ms": t * 1e3, "TFLOP/s": fl / t / 1e12, "hbm_GB/s": (wbytes + abytes) / t / 1e9,
        "hbm_frac": (wbytes + abytes) / t / 1e9 / peaks["hbm_gbs"],
        "roofline_ms": roof_t * 1e3, "frac_of_roofline": roof_t / t,
        "bytes_per_launch": wbytes + abytes, "flops_per_launch": fl,
        "traffic_bytes_per_launch": profiled_traffic("gemm_grouped_moe.md", "gemm_kernel.cuh"),
        "timed": "alone, back to back, mean of the middle 12 of 20 (weights 3.76 GB > L2)"}
    del qa, sa, qw, sw, C, w
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9, 10])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--extras", choices=["all", "none"], default="all",
                    help="none: skip the kernels timed at other shapes and the cuBLAS FP8 ceiling "
                         "(for profiler runs)")
    ap.add_argument("--experts", type=int, default=0,
                    help="MoE configs: keep this many experts (same tokens per expert)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks, peak_kind = load_peaks()

    w = make_workload(args.config, device, args.experts)
    path = make_path(w, device)
    flops = path.flops
    stream = torch.cuda.current_stream()

    clocks = ClockSampler(device)
    clocks.__enter__()
    h_warm = time.perf_counter()
    for _ in range(args.warmup):
        path.step()
    torch.cuda.synchronize()
    assert path.fp8q.fp8q_get_device_status() == 0

    nev = 1 + len(path.names)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    h_start = time.perf_counter()
    start.record(stream)
    for i in range(args.steps):
        path.step(events=events[i])
    stop.record(stream)
    torch.cuda.synchronize()
    h_stop = time.perf_counter()
    if dist is not None:
        dist.barrier()
    elapsed = max_over_ranks(start.elapsed_time(stop) / 1e3, dist, device)
    status = path.fp8q.fp8q_get_device_status()
    clk_timed = clocks.summary(h_start, h_stop)
    clk_timed["window"] = "timed region"
    clk_span = clocks.summary(h_warm, h_stop)
    clk_span["window"] = "warm-up + timed region"

    # per-kernel averages from the events around each launch
    per = {n: statistics.fmean(ev[j].elapsed_time(ev[j + 1]) for ev in events) / 1e3
           for j, n in enumerate(path.names)}
    kern = path.kernels(per)
    for v in kern.values():
        if "GB/s" in v:
            v["frac_hbm"] = v["GB/s"] / peaks["hbm_gbs"]
    # the quantizers again, each launched alone (after the timed region)
    quant_names = [n for n in path.names if n not in path.gemm_names]
    alone = time_alone(path, quant_names, device)
    kern_alone = path.kernels({n: alone.get(n, per[n]) for n in path.names})
    for n in quant_names:
        k = n if n in kern else next(k for k in kern if k.startswith(n))  # quant_act+dispatch
        kern[k]["alone_ms"] = alone[n] * 1e3
        kern[k]["alone_GB/s"] = kern_alone[k]["GB/s"]
        kern[k]["alone_frac_hbm"] = kern_alone[k]["GB/s"] / peaks["hbm_gbs"]

    # the FP8 tensor ceiling of this GPU (cuBLAS, reported beside the GEMM)
    # and the roofline of the dominant kernel, the GEMM(s) (the weight-
    # gradient GEMM in the backward step). The denominator is the larger of
    # the measured FP8 ceiling and 2 x the measured bf16 peak (the nominal
    # FP8:BF16 ratio), in its burst form when the timed region is short and
    # ran without a power cap, else in its sustained form.
    extra = {}
    if args.config == 3 and rank == 0 and world == 1 and args.extras == "all":
        extra = extra_legs(device, peaks)
    fp8 = fp8_ceiling(device, clocks) if rank == 0 and args.extras == "all" else {}
    clocks.__exit__(None, None, None)
    t_gemm = sum(per[n] for n in path.gemm_names)
    t_dom = sum(per[n] for n in path.dominant)
    gemm_tflops = path.dominant_flops / t_dom / 1e12
    fp8_peak, burst_peak, sus_peak, peak_source = choose_fp8_peak(fp8, peaks, peak_kind, elapsed, clk_timed)
    traffic = None
    kernel_profiles = {}
    if args.config == 3:
        traffic = profiled_traffic("gemm_dense_8192x7168x7168.md", "gemm_kernel.cuh")
        kernel_profiles = {"quant_act": ("quant_act_8192x7168.md", "quant.cu"),
                           "quant_weight[B]": ("quant_weight_7168x7168.md", "quant.cu")}
    elif args.config == 9:
        traffic = profiled_traffic("gemm_ue8m0_dense_8192x7168x7168.md", "gemm_bs.cu")
        kernel_profiles = {"quant_act": ("quant_ue8m0_8192x7168.md", "quant.cu")}
    elif args.config == 8:
        traffic = profiled_traffic("gemm_wgrad_7168x7168x8192.md", "gemm_kernel.cuh")
        kernel_profiles = {"quant_act[dY]": ("quant_act_8192x7168.md", "quant.cu"),
                           "quant_weight_t[W]": ("quant_weight_t_7168x7168.md", "quant.cu"),
                           "gemm[dX]": ("gemm_dense_8192x7168x7168.md", "gemm_kernel.cuh"),
                           "quant_act_t[dY]": ("quant_act_t_8192x7168.md", "quant.cu"),
                           "quant_act_t[X]": ("quant_act_t_8192x7168.md", "quant.cu")}
    for kname, (prof, src_file) in kernel_profiles.items():
        kern[kname]["traffic_bytes_per_launch"] = profiled_traffic(prof, src_file)
    roofline = {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": gemm_tflops / fp8_peak, "traffic": traffic,
                "traffic_unit": "DRAM bytes per launch (ncu, profiles/)",
                "frac_of_burst_peak": gemm_tflops / burst_peak,
                "frac_of_sustained_peak": gemm_tflops / sus_peak,
                "frac_of_nominal": gemm_tflops / NOMINAL_FP8_TFLOPS,
                "kernel": ("fp8_gemm_bs_kernel " if getattr(path, "ue8m0", False) else "fp8_gemm_kernel ")
                          + "+".join(path.dominant), "peak_source": peak_source}
    if len(path.dominant) > 1:
        roofline["achieved_over"] = "+".join(path.dominant) + " (total GEMM FLOPs / total GEMM time)"
    if w.offsets is not None:
        # the grouped GEMM streams every expert's weights once: HBM-bound
        M = w.A.shape[0]
        wbytes = w.weights["W"].numel() + 4 * w.weights["W"].numel() // 16384
        abytes = M * w.A.shape[1] + 2 * M * w.weights["W"].shape[1]
        roofline["hbm_GB/s"] = (wbytes + abytes) / t_gemm / 1e9
        roofline["hbm_frac"] = roofline["hbm_GB/s"] / peaks["hbm_gbs"]
    kern.update(extra)

    ms_per_step = elapsed / args.steps * 1e3
    value = job_throughput(world, flops, args.steps, elapsed)

    # end to end through the public API: every step copies its bf16 inputs
    # from pinned host memory and its outputs back to pinned host memory.
    # Two buffer sets and three streams let the copy-in of step i+1 and the
    # copy-out of step i-1 overlap the compute of step i (PCIe is full
    # duplex); events order each buffer's reuse.
    e2e = None
    if args.e2e_steps > 0:
        hostI = {n: t.cpu().pin_memory() for n, t in path.inputs().items()}
        hostO = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory()
                 for n, t in path.outputs().items()}
        devI = [{n: torch.empty_like(t) for n, t in path.inputs().items()} for _ in range(2)]
        devO = [{n: torch.empty_like(t) for n, t in path.outputs().items()} for _ in range(2)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
        ev = lambda: torch.cuda.Event()
        in_done = [ev(), ev()]
        cmp_done = [ev(), ev()]
        out_done = [ev(), ev()]
        def e2e_run(n):
            for i in range(n):
                b = i & 1
                s_in.wait_event(cmp_done[b])         # step i-2 no longer reads buffer b
                with torch.cuda.stream(s_in):
                    for nm in hostI:
                        devI[b][nm].copy_(hostI[nm], non_blocking=True)
                in_done[b].record(s_in)
                s_cmp.wait_event(in_done[b])
                s_cmp.wait_event(out_done[b])       # output buffer b has been copied out
                path.step(inp=devI[b], outs=devO[b], stream=s_cmp)
                cmp_done[b].record(s_cmp)
                s_out.wait_event(cmp_done[b])
                with torch.cuda.stream(s_out):
                    for nm in hostO:
                        hostO[nm].copy_(devO[b][nm], non_blocking=True)
                out_done[b].record(s_out)
        e2e_run(3)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(s_in)
        e2e_run(args.e2e_steps)
        s_in.wait_stream(s_out)
        s1.record(s_in)
        torch.cuda.synchronize()
        te = max_over_ranks(s0.elapsed_time(s1) / 1e3, dist, device)
        e2e = {"value": job_throughput(world, flops, args.e2e_steps, te), "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in hostI.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in hostO.values()),
               "ms_per_step": te / args.e2e_steps * 1e3,
               "pipelined": "copy-in / compute / copy-out on three streams, double-buffered"}

    cpu = None
    if rank == 0 and world == 1:
        threads = os.cpu_count() or 1
        full, desc = sample_oracle(w, 0, threads)
        cpu = {"value": flops / full / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc}

    if rank == 0:
        clk = clk_timed if clk_timed["samples"] > 0 else clk_span
        if clk["sm_mhz"]:
            clk["cycles_per_step"] = ms_per_step * 1e-3 * clk["sm_mhz"] * 1e6
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "e4m3*e4m3->f32", "data": "synthetic",
                "config": run_config(w, world),
                "roofline": roofline, "kernels": kern, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": path.launches_per_step * args.steps,
                "clocks": clk, "clocks_warmup_and_timed": clk_span, "device_status": status,
                "peaks": {"source": peak_kind, "hbm_gbs": peaks["hbm_gbs"],
                          "fp8_burst_tflops": burst_peak, "fp8_sustained_tflops": sus_peak,
                          "fp8_ceiling_measured": fp8, "fp8_nominal_tflops": NOMINAL_FP8_TFLOPS}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
