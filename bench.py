"""Benchmark of the routed MXFP4 MoE layer (one JSON line on stdout, rank 0).

A step is one forward of the whole layer (router, permute, expert FFN, combine) over one batch
of the workload's seeded synthetic tokens. `value` is whole-job tokens/s with inputs already in
HBM; `e2e` is the same metric through coli_moe_forward_host with pinned host buffers (the
host->device copy of x and the device->host copy of out inside the timed region). L2 is flushed
(a 512 MiB write) before every timed step; each step is timed with CUDA events on the layer's
stream, and the L2 flush is outside the events.

--impl reference times the plain-C oracle on the host cores on the same workload (the reference
arm; one oracle forward of a bounded token sample per step).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
Under torchrun every rank runs an independent replica (no collective on the data path).

Other lines (same contract, their own metric or config):
  --format nvfp4          the layer with NVFP4 experts (coli_moe_forward_nvfp4)
  --bank S                routed experts in page-locked host memory behind S device slots, a new
                          token batch every step (roofline: the refill against the measured
                          host-to-device copy rate)
  --dense NAME            the FP8 E4M3 dense projection (coli_dense_forward) on a dense workload
  --ffn-path P            force one FFN path of coli_moe_forward (path comparisons)
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routed_moe_fp4_gb300 import synthetic as S  # noqa: E402

DEFAULT_WORKLOAD = "decode"
METRIC = "MoE-layer tokens/s at 1 GB300"
L2_FLUSH_BYTES = 512 << 20
L2_FLUSH_NOTE = ("flushed before every timed step: a 512 MiB write, then a read of its first 256 MiB, so the "
                 "flush's own dirty lines are written back before the timed region")


def l2_flusher(buf, stream, read: bool = True):
    """A function that evicts the L2 on `stream`: a write of `buf` (larger than the L2) and, with
    `read`, a read of its first half. The write alone leaves the L2 full of dirty lines whose
    write-back then lands inside the next timed region: measured on the decode layer, 173.7 against
    161.4 us per step, the difference being that write-back, not the layer's work."""
    import torch
    half = buf[: buf.numel() // 2]
    sink = torch.empty(1, dtype=buf.dtype, device=buf.device)

    def flush():
        with torch.cuda.stream(stream):
            buf.fill_(1.0)
            if read:
                torch.sum(half, dim=0, keepdim=True, out=sink)
    return flush


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # the timed region starts once nvidia-smi reports (its first query takes a while)
        t0 = time.perf_counter()
        while not self.lines and self.proc.poll() is None and time.perf_counter() - t0 < 3.0:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlPoller:
    """Polls the SM clock and the clock-event reasons through NVML's read-only queries every
    millisecond. A timed region of a few milliseconds falls between two of nvidia-smi's 100 ms
    samples; this poller sees it. Sets nothing on the GPU."""
    NVML_CLOCK_SM = 1
    # clock-event reason bits of nvml.h that slow the clocks (idle, application-clock setting,
    # sync boost and display setting are left out)
    REASONS = ((0x4, "sw_power_cap"), (0x8, "hw_slowdown"), (0x20, "sw_thermal_slowdown"),
               (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"))

    def __init__(self, device_ids, lib=None, period_s: float = 0.001):
        """device_ids: candidates to find the GPU by, tried in order, each ("uuid", "GPU-..."),
        ("pci", "00000000:01:00.0") or ("index", n)."""
        self.ids = list(device_ids)
        self.lib = lib
        self.period = period_s
        self.handle = None
        self.samples = []
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None

    def start(self) -> bool:
        import ctypes as C
        try:
            if self.lib is None:
                self.lib = C.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            h = C.c_void_p()
            for kind, v in self.ids:
                if kind == "uuid":
                    rc = self.lib.nvmlDeviceGetHandleByUUID(v.encode(), C.byref(h))
                elif kind == "pci":
                    rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(v.encode(), C.byref(h))
                else:
                    rc = self.lib.nvmlDeviceGetHandleByIndex_v2(C.c_uint(int(v)), C.byref(h))
                if rc == 0:
                    self.handle = h
                    break
            if self.handle is None:
                raise OSError("no NVML handle for the device")
            mx = C.c_uint()
            if self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM, C.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError) as e:
            self.error = str(e).splitlines()[0][:120] if str(e) else type(e).__name__
            self.handle = None
            return False
        self._thread = threading.Thread(target=self._poll, daemon=True)
        self._thread.start()
        return True

    def _poll(self):
        import ctypes as C
        clk, rs = C.c_uint(), C.c_ulonglong()
        while not self._stop.is_set():
            ok_c = self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, C.byref(clk)) == 0
            ok_r = self._reasons(self.handle, C.byref(rs)) == 0
            if ok_c:
                self.samples.append((float(clk.value), int(rs.value) if ok_r else 0))
            time.sleep(self.period)

    def stop(self):
        """The clock record of the polled window, or None when NVML was not usable."""
        if self._thread is None:
            return None
        self._stop.set()
        self._thread.join(timeout=2)
        try:
            self.lib.nvmlShutdown()
        except AttributeError:
            pass
        if not self.samples:
            return None
        bits = 0
        for _, r in self.samples:
            bits |= r
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz if self.max_mhz else max(c for c, _ in self.samples),
                "sm_min_mhz": min(c for c, _ in self.samples),
                "reasons": [n for b, n in self.REASONS if bits & b], "samples": len(self.samples)}


def nvml_ids(device: int):
    """Ways to find CUDA device `device` in NVML (whose numbering can differ from CUDA's)."""
    import torch
    ids = []
    p = torch.cuda.get_device_properties(device)
    u = str(getattr(p, "uuid", "") or "")
    if u:
        ids.append(("uuid", u if u.startswith("GPU-") else "GPU-" + u))
    if hasattr(p, "pci_bus_id"):
        ids.append(("pci", f"{getattr(p, 'pci_domain_id', 0):08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"))
    ids.append(("index", device))
    return ids


class Clocks:
    """The clock record of a timed region: NVML polled every millisecond inside the region, and
    the nvidia-smi query line of the profiling recipe beside it (100 ms samples)."""

    def __init__(self, device: int, nvml_lib=None, smi: bool = True, ids=None):
        self.smi = ClockSampler(device) if smi else None
        self.device = device
        self.nvml_lib = nvml_lib
        self.ids = ids
        self.nvml = None

    def start(self):
        if self.smi is not None:
            self.smi.start()
        try:
            ids = self.ids if self.ids is not None else nvml_ids(self.device)
        except (RuntimeError, AssertionError, AttributeError):
            ids = [("index", self.device)]
        self.nvml = NvmlPoller(ids, lib=self.nvml_lib)
        self.nvml.start()

    def stop(self) -> dict:
        # NVML first: its window closes with the timed region (nvidia-smi's stop waits 0.25 s)
        nv = self.nvml.stop() if self.nvml is not None else None
        smi = self.smi.stop() if self.smi is not None else None
        if nv is None:
            out = dict(smi or {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"]})
            out["source"] = "nvidia-smi, 100 ms samples" + (
                f" (NVML: {self.nvml.error})" if self.nvml is not None and self.nvml.error else "")
            return out
        reasons = set(nv["reasons"])
        if smi:
            reasons |= {r for r in smi.get("reasons", []) if r != "nvidia-smi unavailable"}
        out = dict(nv, reasons=sorted(reasons), source="NVML every 1 ms inside the timed region")
        if smi:
            out["smi"] = smi
        return out


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# FFN paths: ABI value, kernel (source file stem), activation terms of x and of h as
# (count, bytes per element), and the arithmetic the path computes in.
FFN_PATHS = {
    "auto": (0, None, None, None, None),
    "gemv": (1, "gemv", None, None, "mxfp4 e2m1 weights dequantised to fp16, fp16 x fp16 FMA, fp32 sums"),
    "mxf4": (2, "gemm_mx4", (4, 0.5), (4, 0.5), "mxfp4 e2m1 x e2m1 activation terms, fp32 accumulate"),
    # the NVFP4 layer (coli_moe_forward_nvfp4) is not an FFN path of coli_moe_forward: no ABI value
    "nvf4": (None, "gemm_mx4", (4, 0.5), (4, 0.5),
             "nvfp4 e2m1 (e4m3 scale per 16, fp32 per matrix) x e2m1 activation terms, fp32 accumulate"),
}
PATH_BY_ABI = {v[0]: k for k, v in FFN_PATHS.items() if v[0] is not None}


def algorithmic_bytes(wl, routing: dict, path: str = "mxf4", group: int = 32) -> dict:
    """Bytes each stage of a block-scaled path must move at least once (touched experts from cnt).

    gate/up: the touched experts' gate and up codes + scales, the activation terms of x (+ scales)
             read, the terms of h (+ scales) written;
    down:    the down codes + scales, the h terms read, y (fp32) written;
    layer:   weights of the touched experts + router weights + x read + out written (the minimum
             any implementation moves)."""
    E, H, I, I_s, T, k = wl.E, wl.H, wl.I, wl.I_s, wl.T, wl.top_k
    cnt = routing["cnt"]
    touched = int((cnt[:E] > 0).sum())
    shared = 1 if I_s > 0 else 0
    Imax = max(I, I_s)
    gu_per = lambda i: 2 * i * (H // 2 + H // group)     # gate+up codes and scales (one per group)
    dn_per = lambda i: H * (i // 2 + i // group)
    rows = T * k + T * shared
    (nx, bx), (nh, bh) = FFN_PATHS[path][2] or (2, 1.0), FFN_PATHS[path][3] or (3, 1.0)
    x_terms = int(nx * rows * (H * bx + H // group))
    h_terms = int(nh * rows * (Imax * bh + Imax // group))
    weights = touched * (gu_per(I) + dn_per(I)) + shared * (gu_per(I_s) + dn_per(I_s))
    gate_up = touched * gu_per(I) + shared * gu_per(I_s) + x_terms + h_terms
    down = touched * dn_per(I) + shared * dn_per(I_s) + h_terms + rows * H * 4
    router = E * H * 4 + T * H * 2 + T * E * 4
    return {"touched_experts": touched, "ffn_gate_up": gate_up, "ffn_down": down, "router": router,
            "layer": weights + E * H * 4 + 2 * T * H * 2}


# FP4 dense tensor rate over bf16 dense, from the nominal per-GPU figures (13.5 and 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0


def algorithmic_flops(wl) -> float:
    """The layer's multiply-adds x 2: gate, up and down (6 H I per row) for T*k routed rows and
    T shared rows, plus the router logits (2 T E H)."""
    return 6.0 * wl.H * (wl.T * wl.top_k * wl.I + wl.T * wl.I_s) + 2.0 * wl.T * wl.E * wl.H


def layer_roofline(layer_bytes: int, flops: float, ms: float, hbm_gbs: float, bf16_tflops: float,
                   peak_kind: str) -> dict:
    """The layer against both rooflines: HBM (its minimum bytes) and the FP4 tensor rate (its
    flops; measured bf16 peak x the nominal FP4/bf16 ratio). frac_combined is
    max(bytes / bandwidth, flops / FP4 peak) / time: whichever bound binds."""
    s = ms * 1e-3
    fp4 = bf16_tflops * FP4_OVER_BF16
    t_hbm, t_tc = layer_bytes / (hbm_gbs * 1e9), flops / (fp4 * 1e12)
    return {"bytes": layer_bytes, "ms": ms, "achieved_gbs": layer_bytes / s / 1e9,
            "frac": layer_bytes / s / 1e9 / hbm_gbs, "flops": flops, "achieved_tflops": flops / s / 1e12,
            "fp4_peak_tflops": fp4, "tensor_frac": flops / s / 1e12 / fp4,
            "frac_combined": max(t_hbm, t_tc) / s, "binding": "hbm" if t_hbm >= t_tc else "tensor",
            "peak_source": f"{peak_kind} hbm_gbs; {peak_kind} bf16_tflops x {FP4_OVER_BF16:g} (nominal FP4/bf16)"}


def profiled_traffic(kernel: str, workload: str, profile: str = "", part: str = "gate_up"):
    """DRAM bytes per launch of `part` (the gate/up launch by default) from a committed ncu summary
    (profiles/<profile>_<workload>.json, profile defaulting to the kernel's source stem), or None
    when the kernel's source has changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{profile or kernel}_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        prof = json.load(f)
    with open(os.path.join(ROOT, "routed_moe_fp4_gb300", "csrc", kernel + ".cu"), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if prof.get("source_sha256") != sha:
        return None
    return prof[part]["dram_read_bytes"] + prof[part]["dram_write_bytes"]


def max_over_ranks(value: float, device=None) -> float:
    """The largest value over all ranks (the timed region ends when the slowest rank ends)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# The other configurations of the scope table, timed beside the headline line in the same run:
# the prefill chunk, the skewed prefill, the batched-decode sweep (with the CUDA-core GEMV beside
# the tensor-core path, for the crossover) and the V4-Pro-sized decode.
CONFIG_PASS = ("prefill", "skewed", *[f"sweep_T{t}" for t in S.SWEEP_T], "v4pro_decode")


def config_target(name: str):
    """(roofline fraction the configuration is judged on, target): the decode shapes against HBM,
    the prefill shapes against max(bytes / bandwidth, flops / FP4 rate)."""
    if name in ("prefill", "skewed"):
        return "frac_combined", 0.50
    return "frac", 0.70


def time_steps(layer, x, out, stream, flush, steps: int, warmup: int, local: int):
    """Device time of `steps` forwards, each after an L2 flush outside its CUDA events, with the
    clocks polled over the timed region. Returns ([ms per step], clock record)."""
    import torch
    for _ in range(warmup):
        flush()
        layer.forward(x, out)
    stream.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    clocks = Clocks(local, smi=False)
    torch.cuda.synchronize()
    clocks.start()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        layer.forward(x, out)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], clocks.stop()


def config_entry(name: str, steps: int, warmup: int, local: int, flush_buf, gemv: bool) -> dict:
    """One configuration: mean and median step time, tokens/s, the layer against its rooflines
    and its target, clocks; with `gemv` the CUDA-core GEMV path timed the same way."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs(name, seed=0)
    wl = inputs.workload
    stream = torch.cuda.Stream()
    layer = cm.MoELayer(inputs, stream=stream)
    x = torch.from_numpy(inputs.x.view(np.int16)).cuda()
    out = torch.empty_like(x)

    flush = l2_flusher(flush_buf, stream)
    hbm_gbs, bf16_tf, kind = _peaks()
    ms, ci = time_steps(layer, x, out, stream, flush, steps, warmup, local)
    routing = layer.routing(wl.T)
    ab = algorithmic_bytes(wl, routing, "mxf4")
    mean = sum(ms) / len(ms)
    lr = layer_roofline(ab["layer"], algorithmic_flops(wl), mean, hbm_gbs, bf16_tf, kind)
    key, target = config_target(name)
    entry = {"workload": f"T={wl.T}, H={wl.H}, E={wl.E}, top_k={wl.top_k}, I={wl.I}, I_s={wl.I_s}, bias {wl.bias}",
             "ms_per_step": mean, "ms_median": statistics.median(ms), "tokens_per_s": wl.T / (mean * 1e-3),
             "touched_experts": ab["touched_experts"],
             "layer_roofline": {k: lr[k] for k in ("bytes", "frac", "flops", "tensor_frac", "frac_combined",
                                                   "binding")},
             "target": {"on": key, "at_least": target, "met": bool(lr[key] >= target)},
             "clocks": {k: ci.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}}
    if gemv:
        layer.set_ffn_path(cm.COLI_FFN_GEMV)
        gms, _ = time_steps(layer, x, out, stream, flush, steps, warmup, local)
        gmean = sum(gms) / len(gms)
        entry["gemv"] = {"ms_per_step": gmean, "frac": ab["layer"] / (gmean * 1e-3) / 1e9 / hbm_gbs}
    layer.close()
    del x, out, layer
    torch.cuda.empty_cache()
    return entry


def run_config_pass(local: int, steps: int = 10, warmup: int = 3) -> dict:
    import torch
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    res = {n: config_entry(n, steps, warmup, local, flush_buf, gemv=n.startswith("sweep_")) for n in CONFIG_PASS}
    sweep = [(int(n[len("sweep_T"):]), e) for n, e in res.items() if n.startswith("sweep_")]
    faster = [t for t, e in sorted(sweep) if e["ms_per_step"] < e["gemv"]["ms_per_step"]]
    res["crossover"] = {"tensor_core_path_faster_from_T": faster[0] if faster else None,
                        "note": "the FP4 tensor-core GEMM against the CUDA-core GEMV, same inputs and routing"}
    return res


def run_ours(args, wl_name: str) -> dict:
    import torch
    import torch.distributed as dist
    from routed_moe_fp4_gb300 import build, colimoe as cm

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    nv = args.format == "nvfp4"
    inputs = S.make_nv_inputs(wl_name) if nv else S.make_inputs(wl_name, seed=0)
    wl = inputs.workload
    stream = torch.cuda.Stream()
    layer = (cm.NvMoELayer if nv else cm.MoELayer)(inputs, stream=stream)
    if args.ffn_path != "auto" and not nv:
        layer.set_ffn_path(FFN_PATHS[args.ffn_path][0])
    x = torch.from_numpy(inputs.x.view(np.int16)).cuda()
    out = torch.empty_like(x)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    x_host = torch.from_numpy(inputs.x.view(np.int16).copy()).pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    l2_flush = l2_flusher(flush, stream)

    # warm-up: the timed steps' sequence, so the flush kernel is loaded before the timed region
    for _ in range(args.warmup):
        l2_flush()
        layer.forward(x, out)
    stream.synchronize()
    launches_per_step = layer.launches()
    path = PATH_BY_ABI[layer.ffn_path()]
    kernel = FFN_PATHS[path][1]

    # timed: device-resident inputs
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = Clocks(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        l2_flush()
        starts[i].record(stream)
        layer.forward(x, out)
        ends[i].record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if ws > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), device="cuda")
    ms_per_step = total_ms / args.steps

    # the same steps after a write-only flush, outside the timed region: its dirty lines are
    # written back inside each step (reported beside the timed number, not instead of it)
    wo_flush = l2_flusher(flush, stream, read=False)
    wo_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(min(args.steps, 20))]
    for a, b in wo_ev:
        wo_flush()
        a.record(stream)
        layer.forward(x, out)
        b.record(stream)
    torch.cuda.synchronize()
    wo_ms = sum(a.elapsed_time(b) for a, b in wo_ev) / len(wo_ev)

    # stage breakdown (profiled forwards, outside the timed region)
    layer.set_profiling(True)
    stage_runs = []
    for _ in range(max(3, min(args.steps, 10))):
        l2_flush()
        layer.forward(x, out)
        stage_runs.append(layer.stage_times())
    layer.set_profiling(False)
    stages = {k: statistics.median([r[k] for r in stage_runs]) for k in stage_runs[0]}

    # the same forward captured once in a CUDA graph and replayed (same buffers; L2 flushed
    # outside the events before every replay)
    graph_info = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer.forward(x, out)
        g.replay()
        stream.synchronize()
        gs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ge = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            l2_flush()
            gs[i].record(stream)
            with torch.cuda.stream(stream):
                g.replay()
            ge[i].record(stream)
        torch.cuda.synchronize()
        g_ms = sum(a.elapsed_time(b) for a, b in zip(gs, ge)) / args.steps
        graph_info = {"value": wl.T * ws / (g_ms * 1e-3), "unit": "tokens/s", "ms_per_step": g_ms}
        del g
    except RuntimeError as e:                  # capture not possible: say so, keep the eager numbers
        graph_info = {"unavailable": str(e).splitlines()[0][:200]}

    # end to end: host buffers through coli_moe_forward_host (the NVFP4 layer: the same copies
    # around coli_moe_forward_nvfp4)
    def host_step():
        if not nv:
            layer.forward_host(x_host, out_host)
            return
        with torch.cuda.stream(stream):
            x.copy_(x_host, non_blocking=True)
            layer.forward(x, out)
            out_host.copy_(out, non_blocking=True)
        stream.synchronize()
    for _ in range(2):
        host_step()
    e2e_ms = []
    for _ in range(args.steps):
        l2_flush()
        stream.synchronize()
        t0 = time.perf_counter()
        host_step()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_step = sum(e2e_ms) / len(e2e_ms)

    routing = layer.routing(wl.T)
    if nv:
        path = "nvf4"
    ab = algorithmic_bytes(wl, routing, path, group=16 if nv else 32)
    hbm_gbs, bf16_tf, peak_kind = _peaks()
    dom = "ffn_gate_up"            # the largest kernel: the FFN GEMM's gate/up launch
    achieved = ab[dom] / (stages[dom] * 1e-3) / 1e9
    traffic = profiled_traffic(kernel, wl.name, "gemm_mx4_nv" if nv else kernel)
    tokens = wl.T * ws
    result = {
        "metric": METRIC, "value": tokens / (ms_per_step * 1e-3), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": FFN_PATHS[path][4],
        "data": "synthetic (seeded SplitMix64; MXFP4 experts, bf16 activations)",
        "config": {"workload": f"{wl.name}: T={wl.T}, H={wl.H}, E={wl.E}, top_k={wl.top_k}, I={wl.I}, "
                               f"I_s={wl.I_s}, " + ("NVFP4 E2M1 + E4M3/16 + fp32 per matrix" if nv
                                                    else "MXFP4 E2M1 + UE8M0/32"), "tokens_per_gpu": wl.T,
                   "ffn_path": path, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": L2_FLUSH_NOTE},
        "roofline": {"kernel": f"{kernel} (gate/up launch)", "bound": "hbm", "achieved": achieved, "peak": hbm_gbs,
                     "unit": "GB/s", "frac": achieved / hbm_gbs, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": ab[dom],
                     "kernel_ms": stages[dom]},
        "layer_roofline": layer_roofline(ab["layer"], algorithmic_flops(wl), ms_per_step, hbm_gbs, bf16_tf,
                                         peak_kind),
        "stages_ms": stages, "touched_experts": ab["touched_experts"],
        # per-step spread of the timed region on this rank (value and ms_per_step use the mean)
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "write_only_flush_ms_per_step": wo_ms,
        "e2e": {"value": tokens / (e2e_step * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_step,
                "h2d_bytes_per_step": int(x_host.numel() * 2), "d2h_bytes_per_step": int(out_host.numel() * 2)},
        "graph": graph_info,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock_info,
    }
    layer.close()
    if ws == 1 and not nv and not args.skip_configs:
        result["configs"] = run_config_pass(local)
    if ws > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def host_link_gbs(nbytes: int = 1 << 30) -> float:
    """Host-to-device copy rate from page-locked memory (copy engines), GB/s: the measured
    denominator of the expert bank's refill traffic."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return 3 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9


def run_bank(args, wl_name: str) -> dict:
    """The layer with its routed experts in page-locked host memory and a bank of --bank device
    slots: each step is one forward over a new batch of tokens (so the routing, and the experts the
    bank must fetch, change from step to step)."""
    import torch
    import torch.distributed as dist
    from routed_moe_fp4_gb300 import build, colimoe as cm

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    inputs = S.make_inputs(wl_name, seed=0)
    wl = inputs.workload
    stream = torch.cuda.Stream()
    layer = cm.MoELayer(inputs, stream=stream)
    host = cm.HostExperts(inputs.experts)
    bank = cm.ExpertBank(layer, args.bank, host)
    if args.copy_blocks:
        bank.set_copy_blocks(args.copy_blocks)
    n = args.warmup + args.steps
    xs = [torch.from_numpy(S.x_batch(0, wl.name, 1 + rank * n + i, wl.T, wl.H).view(np.int16)).cuda()
          for i in range(n)]
    out = torch.empty_like(xs[0])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    l2_flush = l2_flusher(flush, stream)

    for i in range(args.warmup):
        l2_flush()
        bank.forward(xs[i], out)
    stream.synchronize()
    before = bank.state()["stats"].copy()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches = 0
    clocks = Clocks(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        l2_flush()
        starts[i].record(stream)
        bank.forward(xs[args.warmup + i], out)
        ends[i].record(stream)
        launches += layer.launches()
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if ws > 1:
        dist.barrier()
    after = bank.state()["stats"]
    ms_per_step = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), device="cuda") / args.steps
    found, copied = int(after[1] - before[1]), int(after[2] - before[2])
    eb = S.expert_bytes(wl.H, wl.I)
    copied_per_step = copied * eb / args.steps

    # end to end: each step's batch from page-locked host memory and its output back to it,
    # inside the timed region (new batches, so the bank sees the same kind of traffic)
    x_hosts = [torch.from_numpy(S.x_batch(0, wl.name, 1 + rank * n + n + i, wl.T, wl.H).view(np.int16)).pin_memory()
               for i in range(args.steps)]
    out_host = torch.empty_like(x_hosts[0]).pin_memory()
    x_dev = torch.empty_like(out)
    e2e_ms = []
    for i in range(args.steps):
        l2_flush()
        stream.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            x_dev.copy_(x_hosts[i], non_blocking=True)
            bank.forward(x_dev, out)
            out_host.copy_(out, non_blocking=True)
        stream.synchronize()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_step = sum(e2e_ms) / len(e2e_ms)
    link = host_link_gbs()
    tokens = wl.T * ws
    result = {
        "metric": METRIC, "value": tokens / (ms_per_step * 1e-3), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": FFN_PATHS["mxf4"][4],
        "data": "synthetic (seeded SplitMix64; MXFP4 experts, bf16 activations; a new token batch every step)",
        "config": {"workload": f"{wl.name}: T={wl.T}, H={wl.H}, E={wl.E}, top_k={wl.top_k}, I={wl.I}, "
                               f"I_s={wl.I_s}, MXFP4 E2M1 + UE8M0/32; routed experts in page-locked host "
                               f"memory, expert bank of {args.bank} device slots",
                   "tokens_per_gpu": wl.T, "ffn_path": "mxf4", "bank_slots": args.bank,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": L2_FLUSH_NOTE},
        "roofline": {"kernel": "bank_refill (experts over the host link)", "bound": "host link",
                     "achieved": copied_per_step / (ms_per_step * 1e-3) / 1e9, "peak": link, "unit": "GB/s",
                     "frac": copied_per_step / (ms_per_step * 1e-3) / 1e9 / link, "traffic": None,
                     "peak_source": "measured in this run: page-locked host-to-device copy (copy engines)",
                     "algorithmic_bytes": copied_per_step},
        "bank": {"slots": args.bank, "found_in_slot": found, "copied": copied,
                 "hit_rate": found / max(1, found + copied), "copied_bytes_per_step": copied_per_step,
                 "copy_blocks": args.copy_blocks or 16},
        "e2e": {"value": tokens / (e2e_step * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_step,
                "h2d_bytes_per_step": int(out_host.numel() * 2), "d2h_bytes_per_step": int(out_host.numel() * 2)},
        "gpu_launches": launches,
        "clocks": clock_info,
    }
    bank.close()
    layer.close()
    if ws > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def run_dense(args, name: str) -> dict:
    """The FP8 dense projection: each step is one projection of the workload's T token rows."""
    import torch
    import torch.distributed as dist
    from routed_moe_fp4_gb300 import build, colimoe as cm

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    inputs = S.make_dense_inputs(name)
    wl = inputs.workload
    stream = torch.cuda.Stream()
    layer = cm.DenseLayer(inputs, stream=stream)
    forced = {"auto": cm.COLI_DENSE_AUTO, "cores": cm.COLI_DENSE_CUDA_CORES, "tensor": cm.COLI_DENSE_TENSOR}[
        args.dense_path]
    layer.set_path(forced)
    x = torch.from_numpy(inputs.x.view(np.int16)).cuda()
    out = torch.empty((wl.T, wl.N), dtype=torch.int16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    l2_flush = l2_flusher(flush, stream)

    for _ in range(args.warmup):
        l2_flush()
        layer.forward(x, out)
    stream.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = Clocks(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        l2_flush()
        starts[i].record(stream)
        layer.forward(x, out)
        ends[i].record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if ws > 1:
        dist.barrier()
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), device="cuda") / args.steps
    assert layer.device_error() == 0
    ran = layer.last_path()

    # both kernel paths forced, outside the timed region (a path that cannot take the shape: null)
    def time_path(path):
        layer.set_path(path)
        try:
            for _ in range(3):
                l2_flush()
                layer.forward(x, out)
        except cm.ColiError:
            return None
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            l2_flush()
            a.record(stream)
            layer.forward(x, out)
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / args.steps
    paths_ms = {"cuda_cores": time_path(cm.COLI_DENSE_CUDA_CORES), "tensor": time_path(cm.COLI_DENSE_TENSOR)}
    layer.set_path(forced)
    assert layer.device_error() == 0

    x_host = torch.from_numpy(inputs.x.view(np.int16).copy()).pin_memory()
    out_host = torch.empty((wl.T, wl.N), dtype=torch.int16).pin_memory()
    e2e = []
    for i in range(args.steps + 2):
        l2_flush()
        stream.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            x.copy_(x_host, non_blocking=True)
            layer.forward(x, out)
            out_host.copy_(out, non_blocking=True)
        stream.synchronize()
        if i >= 2:
            e2e.append((time.perf_counter() - t0) * 1e3)
    e2e_ms = sum(e2e) / len(e2e)

    hbm_gbs, bf16_tf, peak_kind = _peaks()
    fp8_tf = 2.0 * bf16_tf                       # nominal FP8 / bf16 dense ratio (4.5 / 2.25)
    nbytes = wl.N * wl.K + 4 * (wl.N // 128) * (wl.K // 128) + 2 * wl.T * wl.K + 2 * wl.T * wl.N
    flops = 2.0 * wl.T * wl.N * wl.K
    t_hbm, t_tc = nbytes / (hbm_gbs * 1e9), flops / (fp8_tf * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes": nbytes}
    else:
        roof = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": fp8_tf, "unit": "TFLOP/s",
                "peak_source": f"{peak_kind} bf16_tflops x 2 (nominal FP8/bf16 ratio)", "algorithmic_flops": flops}
    cores = ran == cm.COLI_DENSE_CUDA_CORES
    roof.update({"kernel": "gemv_fp8 (one launch)" if cores else "gemm_fp8 (with its activation split)",
                 "frac": roof["achieved"] / roof["peak"],
                 "traffic": profiled_traffic("gemv_fp8", name, part="launch") if cores else None, "kernel_ms": ms})
    tokens = wl.T * ws
    res = {
        "metric": "FP8 dense projection tokens/s at 1 GB300", "value": tokens / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 weights x bf16 activations on the CUDA cores, exact fp32 products, fp32 accumulate"
                  if cores else "e4m3 weights x two e4m3 activation terms, fp32 accumulate, fp32 block-scale folding"),
        "data": "synthetic (seeded SplitMix64; E4M3 weights with fp32 128x128 block scales, bf16 activations)",
        "config": {"workload": f"{wl.name}: T={wl.T}, K={wl.K}, N={wl.N}, E4M3 + fp32 scale per 128x128",
                   "tokens_per_gpu": wl.T, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": L2_FLUSH_NOTE, "path": "cuda cores" if cores else "tensor cores",
                   "path_choice": "forced" if args.dense_path != "auto" else "automatic"},
        "roofline": roof,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(x_host.numel() * 2), "d2h_bytes_per_step": int(out_host.numel() * 2)},
        "gpu_launches": (1 if cores else 2) * args.steps,
        "clocks": clock_info,
        "paths_ms": paths_ms,
    }
    if not args.skip_cpu and rank == 0:
        from oracle.oracle import Oracle
        o = Oracle()
        rows, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_budget:
            o.fp8_linear(inputs.x[: min(8, wl.T)], inputs.w, inputs.w_scale)
            rows += min(8, wl.T)
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": rows / el, "unit": "tokens/s", "cores": o.threads(), "kind": "oracle",
                               "sample": f"{rows} token rows of {wl.name} through the oracle, {el:.1f} s"}
    layer.close()
    if ws > 1:
        dist.destroy_process_group()
    return res if rank == 0 else None


def oracle_sample(wl_name: str, budget_s: float):
    """Times the oracle's full forward on the workload's tokens, repeated up to `budget_s`."""
    from oracle.oracle import Oracle
    inputs = S.make_inputs(wl_name, seed=0)
    wl = inputs.workload
    o = Oracle()
    n_tok, runs = 0, 0
    t0 = time.perf_counter()
    while True:
        o.moe_forward(inputs.x, inputs.router_w, inputs.router_b, wl.top_k, inputs.experts, inputs.shared)
        n_tok += wl.T
        runs += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    res = {"value": n_tok / el, "unit": "tokens/s", "cores": o.threads(), "kind": "oracle",
           "sample": f"{runs} full oracle forward(s) of the {wl.name} workload ({wl.T} tokens each), "
                     f"{el:.1f} s", "cpu_model": cpu_model()}
    # the same oracle built without OpenMP, on one core, for a third of the budget
    o1 = Oracle(openmp=False)
    n1, t1 = 0, time.perf_counter()
    while True:
        o1.moe_forward(inputs.x, inputs.router_w, inputs.router_b, wl.top_k, inputs.experts, inputs.shared)
        n1 += wl.T
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 3:
            break
    res["single_thread"] = {"value": n1 / el1, "unit": "tokens/s", "cores": 1,
                            "sample": f"{n1 // wl.T} forward(s), {el1:.1f} s"}
    return res


# Arm CPU part numbers (MIDR_EL1 PartNum, implementer 0x41) of the cores these hosts carry.
_ARM_PARTS = {0xD40: "Neoverse-V1", 0xD49: "Neoverse-N2", 0xD4F: "Neoverse-V2", 0xD83: "Neoverse-V3",
              0xD8E: "Neoverse-N3"}


def cpu_model(cpuinfo: str = "/proc/cpuinfo") -> str:
    """The host CPU's model: the "model name" line of /proc/cpuinfo where there is one (x86), else
    `lscpu`'s "Model name", else the Arm implementer and part number (Grace: Neoverse-V2), else the
    machine type."""
    import platform
    import subprocess
    fields = {}
    try:
        with open(cpuinfo) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    for key in ("model name", "cpu model", "hardware"):
        if fields.get(key):
            return fields[key]
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                name = line.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        impl, part = int(fields["cpu implementer"], 16), int(fields["cpu part"], 16)
        name = _ARM_PARTS.get(part, f"part 0x{part:03x}") if impl == 0x41 else f"implementer 0x{impl:02x} part 0x{part:03x}"
        return f"Arm {name}" if impl == 0x41 else name
    except (KeyError, ValueError):
        pass
    return platform.machine()


def run_reference(args, wl_name: str):
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    from oracle.oracle import Oracle
    inputs = S.make_inputs(wl_name, seed=0)
    wl = inputs.workload
    o = Oracle()
    fwd = lambda: o.moe_forward(inputs.x, inputs.router_w, inputs.router_b, wl.top_k, inputs.experts,
                                inputs.shared)
    for _ in range(args.warmup):
        fwd()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fwd()
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    v = wl.T / (ms * 1e-3)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.name}: T={wl.T}, H={wl.H}, E={wl.E}, top_k={wl.top_k}, I={wl.I}, "
                                   f"I_s={wl.I_s}, MXFP4 E2M1 + UE8M0/32"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": o.threads(), "kind": "oracle",
                             "sample": f"{args.steps} timed full oracle forwards of {wl.T} tokens"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(S.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--skip-cpu", action="store_true", help="no cpu_baseline (profiling runs)")
    ap.add_argument("--skip-configs", action="store_true",
                    help="no per-configuration pass beside the headline line (profiling runs)")
    ap.add_argument("--ffn-path", default="auto", choices=sorted(PATH_BY_ABI.values()),
                    help="force an FFN path (default: the library's own choice)")
    ap.add_argument("--format", default="mxfp4", choices=["mxfp4", "nvfp4"],
                    help="expert weight format of the MoE layer (nvfp4: the format variant)")
    ap.add_argument("--bank", type=int, default=0,
                    help="routed experts in page-locked host memory behind a bank of this many device slots")
    ap.add_argument("--copy-blocks", type=int, default=0, help="bank: blocks that copy while a round computes")
    ap.add_argument("--dense", default="", choices=[""] + sorted(S.DENSE_WORKLOADS),
                    help="time the FP8 dense projection on this workload instead of the MoE layer")
    ap.add_argument("--dense-path", default="auto", choices=["auto", "cores", "tensor"],
                    help="FP8 projection: force the CUDA-core or the tensor-core kernel path")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        res = run_reference(args, args.workload)
    else:
        if args.dense:
            res = run_dense(args, args.dense)
            args.skip_cpu = True                 # run_dense times its own oracle sample
        else:
            res = run_bank(args, args.workload) if args.bank else run_ours(args, args.workload)
        if res is not None and not args.skip_cpu:
            res["cpu_baseline"] = oracle_sample(args.workload, args.cpu_budget)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
