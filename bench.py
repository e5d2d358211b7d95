"""Benchmark of the deterministic, batch-invariant linear-logp (and det_gemm) on GB300.

Default line: fused linear-logp on N=4096 rows, H=4096, V=151936 (BF16 operands,
FP32 accumulation, no bias, uniform int64 targets, seeded synthetic data).  One
step = the whole operator: the fused projection + online-softmax kernel and the
split-merge kernel, on inputs resident in HBM.  The weight (1.245 GB) is larger
than the 129 MB L2, so every step streams it from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mid|large|det_gemm]
  python bench.py --impl reference ...     # the FP64 CPU oracle on the host cores

Printed: one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (the operator needs no
exchange between GPUs); the timed region is bracketed by a barrier and the
slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "linear-logp tokens/s & TFLOP/s (N=4096,H=4096,V=151936); % BF16 dense peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- measured traffic
# The source files each recorded kernel is built from (its translation unit and the
# headers that define its loops, schedule and launch).
_COMMON = ["rlk_device.cuh", "rlk_pipeline.cuh", "rlk_internal.h", "common.cu"]
KERNEL_SOURCES = {
    "linear_logp_partials_kernel": _COMMON + ["rlk_solo.cuh", "linear_logp.cu"],
    "linear_logp_solo_kernel": _COMMON + ["rlk_solo.cuh", "linear_logp.cu"],
    "det_gemm_kernel": _COMMON + ["det_gemm.cu"],
}


def kernel_sources_sha256(kernel: str) -> str:
    """Hash of the code of the files `kernel` is built from: comments and whitespace
    are dropped, so editing a comment does not invalidate the recorded captures."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deterministic_invariant_gemm_linear_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture, or None when there is
    none for this kernel / workload or the kernel's sources changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{kernel}@{workload}")
    if not rec or rec.get("sources_sha256") != kernel_sources_sha256(kernel):
        return None
    return rec["dram_bytes_per_launch"]


# ---------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        rank = dist.get_rank()
        local = int(os.environ.get("LOCAL_RANK", rank))
        return rank, world, local
    return 0, 1, 0


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
# NVML clock-event reason bits (nvml.h): read only, never set.
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """Read-only NVML queries through ctypes (the NVIDIA driver's libnvidia-ml): the SM
    clock, its maximum and the active clock-event reasons."""

    def __init__(self, device: torch.device):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:   # match the CUDA device to its NVML handle by PCI bus id
            p = torch.cuda.get_device_properties(device)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
            ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) == 0
        except (AttributeError, TypeError):
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(
                ctypes.c_uint(device.index or 0), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        v = ctypes.c_uint()
        self.max_mhz = float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.h, 1, ctypes.byref(v)) == 0 else None

    def sample(self):
        c = self.c
        clk, rs = c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(clk)) != 0:   # NVML_CLOCK_SM
            return None
        reasons = rs.value if self.reasons_fn(self.h, c.byref(rs)) == 0 else 0
        return float(clk.value), reasons


class ClockSampler:
    """SM clock / throttle-reason samples taken while the timed region runs: NVML
    every ~2 ms from a thread of this process (read-only queries), else
    nvidia-smi every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device if isinstance(device, torch.device) else torch.device("cuda", device)
        self.proc = None
        self.nvml = None
        self.lines = []
        self.samples = []
        self.stop = threading.Event()
        self.thread = None

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.device)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _poll(self):
        while not self.stop.is_set():
            s = self.nvml.sample()
            if s is not None:
                self.samples.append(s)
            self.stop.wait(0.002)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        if self.nvml is not None:
            if not self.samples:
                return None
            sm = [x[0] for x in self.samples]
            reasons = set()
            for _, r in self.samples:
                reasons.update(n for bit, n in _NVML_REASONS.items() if r & bit)
            return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": self.nvml.max_mhz,
                    "sm_mhz_min": min(sm), "sm_mhz_max": max(sm), "reasons": sorted(reasons),
                    "samples": len(sm), "source": "NVML in-process, ~2 ms period"}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 50 ms period"}


# Dense BF16 tensor-core rate per SM per clock on this architecture: one
# M=128 x N=256 x K=16 MMA (1,048,576 FLOP) per 128 cycles, i.e. 8192 FLOP/clk
# (the nominal 2.25 PFLOP/s over 152 SMs corresponds to ~1.81 GHz).
BF16_FLOP_PER_SM_CLK = 8192


def per_clock(achieved_tflops: float, clocks, device) -> dict:
    """The achieved rate normalised by the SM clock sampled during the timed region."""
    if not clocks or not clocks.get("sm_mhz"):
        return {}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = clocks["sm_mhz"]
    ceiling = sms * BF16_FLOP_PER_SM_CLK * mhz * 1e6 / 1e12
    return {"tflops_per_ghz": achieved_tflops / (mhz / 1e3),
            "per_clock_ceiling_tflops": ceiling,
            "per_clock_frac": achieved_tflops / ceiling,
            "per_clock_note": f"{sms} SMs x {BF16_FLOP_PER_SM_CLK} dense BF16 FLOP/clk x median "
                              f"{mhz:.0f} MHz as NVML reports it; the SMs' own cycle counters read "
                              "8-20% lower under tensor load (profiles/"
                              "linear_logp_partials_effective_clock.md), so this understates the "
                              "work per actual cycle"}


# ---------------------------------------------------------------- CPU oracle leg
def oracle_gemm_tflops(A, B, dC, rows: int):
    """Time the FP64 oracle's fwd, dA and dB on `rows` output rows each (host cores)."""
    import oracle
    orc = oracle.load()
    cores = orc.max_threads()
    a, b, d = si.bf16_bits(A), si.bf16_bits(B), si.bf16_bits(dC)
    r = np.arange(rows, dtype=np.int64)
    t0 = time.perf_counter()
    orc.gemm_fwd(a, b, rows=r, threads=cores)
    orc.gemm_da(d, b, rows=r, threads=cores)
    orc.gemm_db(a, d, rows=r, threads=cores)
    dt = time.perf_counter() - t0
    flop = 2.0 * rows * (B.shape[1] * A.shape[1] + dC.shape[1] * B.shape[0] + dC.shape[1] * A.shape[0])
    return flop / dt / 1e12, dt, cores


def oracle_tokens_per_s(hidden, weight, target, bias, rows: int):
    """Time the FP64 oracle on `rows` rows of the workload (host cores)."""
    import oracle
    orc = oracle.load()
    cores = min(orc.max_threads(), rows)
    hb, wb = si.bf16_bits(hidden[:rows]), si.bf16_bits(weight)
    tb = target[:rows].cpu().numpy()
    bb = None if bias is None else bias.cpu().numpy()
    t0 = time.perf_counter()
    orc.linear_logp(hb, wb, tb, bb, threads=cores)
    dt = time.perf_counter() - t0
    return rows / dt, dt, cores


# ---------------------------------------------------------------- L2 flush
def flush_l2(buf: torch.Tensor):
    """Evict the L2 before a cold-cache step: write a buffer larger than the L2
    (256 MB > 129 MB), then read it back, so the lines left behind are clean and the
    timed kernel does not pay for writing the flush's dirty lines back to HBM."""
    buf.zero_()
    buf.view(torch.int64).sum()


# ---------------------------------------------------------------- workloads
def linear_logp_metric(w) -> str:
    return f"linear-logp tokens/s & TFLOP/s (N={w.N},H={w.H},V={w.V}); % BF16 dense peak"


def linear_logp_config(w, world: int) -> dict:
    """The `config` of a linear-logp line: the same for the GPU arm and the reference arm."""
    w_bytes = w.V * w.H * 2
    return {"workload": f"{w.name}: N={w.N} H={w.H} V={w.V}" + (" +bias" if w.bias else "")
            + ", hidden~N(0,1), W~N(0,1/sqrt(H)), uniform int64 targets, seed=rank",
            "global_batch": w.N * world, "seq_len": None, "parallelism": f"replicas x{world}",
            "l2": (f"inputs larger than L2: W {w_bytes / 1e9:.3f} GB streamed per step"
                   if w_bytes >= (512 << 20) else "L2 flushed (256 MB write, then read) before every "
                   "step; step time = sum of per-step kernel events")}


def linear_logp_bench(args, dev, rank, world, peaks, peak_src):
    import deterministic_invariant_gemm_linear_gb300 as rlk
    if args.workload == "ragged":
        w = si.ragged(args.rows or 17)
    else:
        w = {"mid": si.MID, "large": si.LARGE, "tiny": si.TINY}[args.workload]
    if args.rows and args.workload != "ragged":
        w = si.LinearLogpWorkload(f"{w.name} (rows={args.rows})", N=args.rows, H=w.H, V=w.V,
                                  bias=w.bias, target_mode=w.target_mode)
    hidden, weight, bias, target = si.workload_inputs(w, seed=rank, device=dev)
    call = rlk.LinearLogpCall(hidden, weight, target, bias)
    stream = torch.cuda.current_stream()
    flops = 2.0 * w.N * w.H * w.V
    # warm-up (untimed)
    for _ in range(args.warmup):
        call.partials()
        call.combine()
    torch.cuda.synchronize()
    K = args.steps
    # W larger than L2 streams from HBM by itself; smaller weights get an L2 flush
    # (a 256 MB write) before every step, outside the per-step kernel events.
    w_bytes = weight.numel() * 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if w_bytes < (512 << 20) else None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clocks:
        start.record(stream)
        for k in range(K):
            if flush is not None:
                flush_l2(flush)
            ev[k][0].record(stream)
            call.partials()
            ev[k][1].record(stream)
            call.combine()
            ev[k][2].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    if flush is None:
        t_local = start.elapsed_time(end) / 1e3
    else:
        t_local = sum(e[0].elapsed_time(e[2]) for e in ev) / 1e3
    t = max_over_ranks(t_local, world, dev)
    assert rlk.device_error() == 0, "device error word set during the bench"
    part_all = [e[0].elapsed_time(e[1]) for e in ev]
    comb_all = [e[1].elapsed_time(e[2]) for e in ev]
    part_ms, comb_ms = float(np.mean(part_all)), float(np.mean(comb_all))
    step_stats = {"partials_median_ms": float(np.median(part_all)), "partials_best_ms": float(min(part_all)),
                  "combine_median_ms": float(np.median(comb_all)), "combine_best_ms": float(min(comb_all))}
    warm = whole = None
    if flush is not None:
        # the same steps with W left in L2 by the previous step (reported beside the cold numbers)
        for k in range(K):
            ev[k][0].record(stream)
            call.partials()
            ev[k][1].record(stream)
            call.combine()
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        warm = {"partials_ms": float(np.mean([e[0].elapsed_time(e[1]) for e in ev])),
                "combine_ms": float(np.mean([e[1].elapsed_time(e[2]) for e in ev])),
                "note": "no flush between steps: W (%.1f MB) partly L2-resident" % (w_bytes / 1e6)}
        # whole calls (partials + combine, no event between them: the combine's launch
        # overlaps the partials kernel's tail), L2 flushed before each as in the timed region
        for k in range(K):
            flush_l2(flush)
            ev[k][0].record(stream)
            call()
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        whole = {"ms": float(np.mean([e[0].elapsed_time(e[2]) for e in ev])),
                 "note": "partials + combine with no event between them (the combine's launch "
                         "overlaps the partials tail), L2 flushed (write, then read) before each call"}
    ms_step = t / K * 1e3
    tokens = w.N * world * K
    value = tokens / t
    S = rlk.vocab_split_policy(w.V)[0]
    alg_bytes = 2 * w.V * w.H + 2 * w.N * w.H + 8 * w.N + 8 * w.N * S + 4 * w.N + (4 * w.V if w.bias else 0)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    hbm_bound = flops / alg_bytes < ridge
    traffic = measured_traffic("linear_logp_solo_kernel" if w.N <= 128 else "linear_logp_partials_kernel",
                               w.name)
    if hbm_bound:
        achieved = alg_bytes / (part_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "peak_kind": f"{peak_src} HBM copy bandwidth",
                "algorithmic": f"{alg_bytes} bytes per launch (W + hidden + targets + partials)"}
    else:
        achieved = flops / (part_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                "peak_kind": f"{peak_src} burst bf16 (sustained {peaks['bf16_tflops_sustained']})",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "algorithmic": f"2*N*H*V = {flops:.4g} FLOP per launch"}
    # calls of at most 128 rows run the one-CTA kernel, larger ones the 2-SM kernel
    roof["kernel"] = "linear_logp_solo_kernel" if w.N <= 128 else "linear_logp_partials_kernel"
    roof["traffic_unit"] = "bytes per launch (ncu dram read+write)"
    peak = peaks["bf16_tflops"]
    line = {
        "metric": linear_logp_metric(w),
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": linear_logp_config(w, world),
        "tflops": flops * world * K / t / 1e12,
        "frac_bf16_peak": flops * K / t_local / 1e12 / peak,
        "kernels_ms": {"linear_logp_partials": part_ms, "linear_logp_combine": comb_ms},
        "kernels_step_stats": step_stats,
        "roofline": roof,
        **({"l2_warm": warm} if warm is not None else {}),
        **({"whole_call": whole} if whole is not None else {}),
        "clocks": clocks.summary(),
        "gpu_launches": 2 * K,
    }
    if roof["bound"] == "tensor":
        roof.update(per_clock(roof["achieved"], line["clocks"], dev))
    if args.phases:
        line["phases"] = phase_breakdown(rlk, call, flush, K, stream, alg_bytes, peaks)
    # ---- e2e through the public API with host buffers (pinned), copies timed.
    if not args.no_e2e:
        line["e2e"] = e2e_linear_logp(w, hidden, weight, target, bias, call, dev, world, K, stream,
                                      copy_weight=False)
        line["e2e_weight_copied_each_step"] = e2e_linear_logp(w, hidden, weight, target, bias,
                                                              call, dev, world, K, stream,
                                                              copy_weight=True)
    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        rows = min(w.N, 2 * oracle.load().max_threads())
        tps, dt, cores = oracle_tokens_per_s(hidden, weight, target, bias, rows)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{rows} rows of the {w.name} workload (full V, full H), "
                                          f"FP64, {dt:.2f} s wall"}
    return line


def e2e_linear_logp(w, hidden, weight, target, bias, call, dev, world, K, stream, copy_weight):
    """Tokens/s through the public binding with host buffers: every step copies its
    activations (hidden, targets) from pinned host memory and reads logp and lse
    back; the lm-head weight (and bias) is model state uploaded once before the
    timed region (copy_weight=False) or, as a bound, copied every step too.
    Two buffer sets alternate, so a step's host-to-device copies (copy stream)
    overlap the previous step's kernels; every step still moves all its bytes
    inside the timed region."""
    import deterministic_invariant_gemm_linear_gb300 as rlk
    hh = hidden.cpu().pin_memory()
    th = target.cpu().pin_memory()
    wh = weight.cpu().pin_memory() if copy_weight else None
    bh = bias.cpu().pin_memory() if (copy_weight and bias is not None) else None
    sets = [(hidden, weight, target, bias, call)]
    h2, t2 = torch.empty_like(hidden), torch.empty_like(target)
    w2 = torch.empty_like(weight) if copy_weight else weight
    b2 = (torch.empty_like(bias) if (copy_weight and bias is not None) else bias)
    sets.append((h2, w2, t2, b2, rlk.LinearLogpCall(h2, w2, t2, b2)))
    outs = [(torch.empty(w.N, dtype=torch.float32).pin_memory(),
             torch.empty(w.N, dtype=torch.float32).pin_memory()) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [None, None]
    E = max(3, min(K, 20))
    for i in range(E + 2):
        b = i % 2
        hd, wd, td, bd, c = sets[b]
        if i == 2:
            torch.cuda.synchronize()
            barrier(world)
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            copy_stream.wait_event(e0)
        if free[b] is not None:
            copy_stream.wait_event(free[b])      # the kernels that last read set b are done
        with torch.cuda.stream(copy_stream):
            hd.copy_(hh, non_blocking=True)
            td.copy_(th, non_blocking=True)
            if copy_weight:
                wd.copy_(wh, non_blocking=True)
                if bd is not None:
                    bd.copy_(bh, non_blocking=True)
        ready[b].record(copy_stream)
        stream.wait_event(ready[b])
        c()
        free[b] = torch.cuda.Event()
        free[b].record(stream)
        outs[b][0].copy_(c.logp, non_blocking=True)
        outs[b][1].copy_(c.lse, non_blocking=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record(stream)
    torch.cuda.synchronize()
    te = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    h2d = hh.numel() * 2 + th.numel() * 8
    if copy_weight:
        h2d += wh.numel() * 2 + (0 if bh is None else bh.numel() * 4)
    return {"value": w.N * world * E / te, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 8 * w.N,
            "ms_per_step": te / E * 1e3, "h2d_gbs": h2d * E / te / 1e9,
            "inputs": ("hidden + targets copied host-to-device every step, logp + lse read back; "
                       "the lm-head weight" + (" and bias" if bias is not None else "") +
                       (" copied every step as well" if copy_weight else
                        " is model state, uploaded once before the timed region")),
            "pipelining": "two buffer sets; a step's host-to-device copies (copy stream) overlap "
                          "the previous step's kernels"}


def role_counters(used, H):
    """The debug trace's role cycle counters (fields 8-15) of one launch, as means over
    the CTAs that recorded them: the MMA issuer's cycles per accumulator tile against
    the tensor-pipe ideal (4 MMAs of 128 cycles per 64-wide reduction block: a pair's
    M=256 x N=256 x K=16 and a single CTA's M=128 x N=256 x K=16 MMA both do 2^20
    FLOP per SM, 8192 dense BF16 FLOP per SM clock), and the fraction of each role's
    cycles spent waiting."""
    mma = used[used[:, 10] > 0]
    load = used[used[:, 13] > 0]
    epi = used[(used[:, 14] + used[:, 15]) > 0]
    if len(mma) == 0:
        return {}
    ideal = -(-H // 64) * 4 * 128
    per_tile = mma[:, 10] / np.maximum(mma[:, 11], 1)
    return {
        "mma_cycles_per_tile": float(per_tile.mean()),
        "mma_ideal_cycles_per_tile": float(ideal),
        "mma_issue_efficiency": float(ideal / per_tile.mean()),
        "mma_operand_wait_frac": float((mma[:, 8] / mma[:, 10]).mean()),
        "mma_accumulator_wait_frac": float((mma[:, 9] / mma[:, 10]).mean()),
        "load_slot_wait_frac": float((load[:, 12] / load[:, 13]).mean()) if len(load) else None,
        "epilogue_wait_frac": float((epi[:, 14] / (epi[:, 14] + epi[:, 15])).mean()) if len(epi) else None,
        "epilogue_work_cycles_per_tile": float((epi[:, 15] / np.maximum(
            mma[:, 11].mean(), 1)).mean()) if len(epi) else None,
    }


def phase_breakdown(rlk, call, flush, K, stream, alg_bytes, peaks):
    """Where a partials launch spends its time, from the debug build's per-CTA phase
    trace (%globaltimer): for K single launches (L2 flushed first when the weight
    fits in it), the times of each phase relative to the first CTA's entry, as the
    median over CTAs and the latest CTA, then the median over launches."""
    if not rlk.is_debug_build():
        raise SystemExit("--phases reads the debug build's trace: run with RLK_LIBRARY=debug")
    names = ["entry", "setup_done", "first_stage_landed", "last_accumulator_complete",
             "last_partials_written", "exit"]
    per = []
    for _ in range(K):
        if flush is not None:
            flush_l2(flush)
        rlk.debug_trace()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call.partials()
        e1.record(stream)
        torch.cuda.synchronize()
        tr = rlk.debug_trace().astype(np.int64)
        used = tr[tr[:, 4] > 0]
        t0 = used[:, 0].min()
        row = {"event_us": e0.elapsed_time(e1) * 1e3, "ctas": int(len(used))}
        # the clock each CTA ran at: SM cycles between entry and exit over the elapsed ns
        cyc = used[:, 7] - used[:, 6]
        ns = used[:, 5] - used[:, 0]
        ok = (cyc > 0) & (ns > 0)
        row["sm_clock_mhz_median"] = float(np.median(cyc[ok] / ns[ok])) * 1e3 if ok.any() else None
        for f, n in enumerate(names):
            v = used[:, f]
            v = v[v > 0] - t0
            row[f"{n}_median_us"] = float(np.median(v)) / 1e3
            row[f"{n}_last_us"] = float(v.max()) / 1e3
        row.update(role_counters(used, call.H))
        per.append(row)
    out = {k: float(np.median([r[k] for r in per if r.get(k) is not None])) for k in per[0]
           if any(r.get(k) is not None for r in per)}
    # the clock under load: the last of K launches run back to back
    rlk.debug_trace()
    for _ in range(K):
        if flush is not None:
            flush_l2(flush)
        call.partials()
    torch.cuda.synchronize()
    tr = rlk.debug_trace().astype(np.int64)
    used = tr[tr[:, 4] > 0]
    cyc, ns = used[:, 7] - used[:, 6], used[:, 5] - used[:, 0]
    ok = (cyc > 0) & (ns > 0)
    out["sm_clock_mhz_under_load"] = float(np.median(cyc[ok] / ns[ok])) * 1e3 if ok.any() else None
    out["span_under_load_us"] = float(used[:, 5].max() - used[:, 0].min()) / 1e3
    out["hbm_floor_us"] = alg_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    out["note"] = ("debug build (store checks on); times from the first CTA's entry; "
                   "event_us - exit_last_us = launch latency and event overhead; mma_* / "
                   "load_* / epilogue_* from the roles' SM cycle counters (the MMA issuer "
                   "runs ahead of the tensor pipe, so its operand waits include time the "
                   "pipe is still busy with MMAs already issued)")
    return out


def backward_bench(args, dev, rank, world, peaks, peak_src):
    """One step = the whole linear-logp backward (grad_hidden + grad_weight) on the mid shape."""
    import deterministic_invariant_gemm_linear_gb300 as rlk
    w = si.MID
    N = args.rows or w.N
    hidden, weight, bias, target = si.workload_inputs(w, seed=rank, device=dev)
    hidden, target = hidden[:N].contiguous(), target[:N].contiguous()
    g = torch.randn(N, generator=torch.Generator(device=dev).manual_seed(7), device=dev)
    _, lse = rlk.linear_logp(hidden, weight, target, bias)
    lib = rlk.lib()
    H, V = w.H, w.V
    ldG = -(-V // 8) * 8
    ws = torch.empty(lib.rlk_linear_logp_backward_workspace_size(N, V), dtype=torch.uint8, device=dev)
    dh = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(V, H, dtype=torch.bfloat16, device=dev)
    sp = rlk._stream_ptr(None)
    P = rlk._ptr

    def step(want_h=True, want_w=True):
        rlk._check(lib.rlk_linear_logp_backward(
            P(hidden), N, H, H, P(weight), V, H, None, P(target), 1, P(lse), P(g),
            P(dh) if want_h else None, rlk.RLK_BF16, H, P(dw) if want_w else None, rlk.RLK_BF16, H,
            None, P(ws), ws.numel(), sp), "rlk_linear_logp_backward")

    def gemm_dh():
        rlk._check(lib.rlk_det_gemm_fwd(P(ws), N, V, ldG, P(weight), H, H, P(dh), rlk.RLK_BF16, H,
                                        None, 0, sp), "rlk_det_gemm_fwd")

    def gemm_dw():
        rlk._check(lib.rlk_det_gemm_db(P(ws), N, V, ldG, P(hidden), rlk.RLK_BF16, H, H, P(dw),
                                       rlk.RLK_BF16, H, None, 0, sp), "rlk_det_gemm_db")

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps

    def timed(fn):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(K):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / 1e3

    barrier(world)
    with ClockSampler(dev) as clocks:
        t_local = timed(step)
    t = max_over_ranks(t_local, world, dev)
    t_dh, t_dw = timed(gemm_dh), timed(gemm_dw)
    t_h_only = timed(lambda: step(want_w=False))          # G kernel + grad_hidden alone
    assert rlk.device_error() == 0
    flop_one = 2.0 * N * H * V
    flops = 3 * flop_one
    t_g = t_h_only - t_dh
    # the library runs both products in one launch when the longer-reduction one
    # fills at most half of the SM pairs, else as two launches
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    long_tiles = -(-min(N, V) // 256) * -(-H // 256)
    one_launch = 2 * long_tiles <= sms // 2
    part = {"grad_logits_kernel (by difference)": t_g / K * 1e3,
            "grad_hidden + grad_weight (by difference; " + ("one launch)" if one_launch else
                                                           "two launches)"): (t_local - t_g) / K * 1e3,
            "grad_hidden det_gemm_fwd alone": t_dh / K * 1e3,
            "grad_weight det_gemm_db alone": t_dw / K * 1e3}
    peak = peaks["bf16_tflops"]
    achieved = flops * K / t_local / 1e12
    line = {
        "metric": f"linear-logp backward TFLOP/s (N={N},H={H},V={V}; grad_hidden + grad_weight)",
        "value": flops * world * K / t / 1e12, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"linear-logp backward: N={N} H={H} V={V}, g~N(0,1), BF16 outputs",
                   "l2": f"inputs larger than L2: W {V * H * 2 / 1e9:.3f} GB and G {N * ldG * 2 / 1e9:.3f} GB per step"},
        "tokens_per_s": N * world * K / t,
        "kernels_ms": part,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "whole backward step (G kernel, then the two products: " +
                               ("one launch)" if one_launch else "two launches)"),
                     "algorithmic": f"3 x 2*N*H*V = {flops:.4g} FLOP per step",
                     "peak_kind": f"{peak_src} burst bf16"},
        "clocks": clocks.summary(),
        "gpu_launches": (2 if one_launch else 3) * K,
    }
    line["roofline"].update(per_clock(line["roofline"]["achieved"], line["clocks"], dev))
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        orc = oracle.load()
        rows = orc.max_threads()
        hb, wb = si.bf16_bits(hidden[:rows]), si.bf16_bits(weight)
        t0 = time.perf_counter()
        orc.linear_logp_backward(hb, wb, target[:rows].cpu().numpy(), g[:rows].cpu().numpy(),
                                 threads=rows)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 3 * 2.0 * rows * H * V / dt / 1e12, "unit": "TFLOP/s",
                                "cores": rows, "kind": "oracle",
                                "sample": f"{rows} rows of the backward (G by definition in FP64, "
                                          f"then float64 products), full V and H, {dt:.2f} s wall"}
    return line


def det_gemm_bench(args, dev, rank, world, peaks, peak_src):
    import deterministic_invariant_gemm_linear_gb300 as rlk
    M = K_ = N = 4096
    A, B, dC = si.det_gemm_inputs(M, K_, N, seed=rank, device=dev)
    flop = 2.0 * M * N * K_
    ops = [("fwd", lambda: rlk.det_gemm_fwd(A, B)), ("da", lambda: rlk.det_gemm_da(dC, B)),
           ("db", lambda: rlk.det_gemm_db(A, dC))]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 256 MB > L2
    for _ in range(args.warmup):
        for _, f in ops:
            f()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    K = args.steps
    per = {n: [] for n, _ in ops}
    total = 0.0
    barrier(world)
    with ClockSampler(dev) as clocks:
        for _ in range(K):
            flush_l2(flush)
            s = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            prev = s
            for n, f in ops:
                f()
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                per[n].append((prev, e))
                prev = e
            torch.cuda.synchronize()
            total += s.elapsed_time(prev) / 1e3
    t = max_over_ranks(total, world, dev)
    ms = {n: float(np.mean([a.elapsed_time(b) for a, b in v])) for n, v in per.items()}
    peak = peaks["bf16_tflops"]
    # cuBLAS bf16 matmul on the same box, as context only
    for _ in range(3):
        torch.matmul(A, B)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(10):
        torch.matmul(A, B)
    c1.record(stream)
    torch.cuda.synchronize()
    cublas = flop / (c0.elapsed_time(c1) / 10 / 1e3) / 1e12
    # the linear layout (weight [N, K]) and the two-product backward, same sizes, as context
    W = B.T.contiguous()
    dC32 = dC.float()
    extra = [("linear_fwd", lambda: rlk.det_linear(A, W)), ("linear_dx", lambda: rlk.det_linear_dx(dC, W)),
             ("linear_dw", lambda: rlk.det_linear_dw(dC, A)),
             ("backward_da_db_bf16_dC", lambda: rlk.det_gemm_backward(dC, A, B)),
             ("da_then_db_bf16_dC", lambda: (rlk.det_gemm_da(dC, B), rlk.det_gemm_db(A, dC))),
             ("backward_da_db_fp32_dC", lambda: rlk.det_gemm_backward(dC32, A, B)),
             ("da_then_db_fp32_dC", lambda: (rlk.det_gemm_da(dC32, B), rlk.det_gemm_db(A, dC32))),
             ("linear_backward_dx_dw_bf16_dY", lambda: rlk.det_linear_backward(dC, A, W))]
    extra_ms = {}
    for name, f in extra:
        f()
        ts = []
        for _ in range(max(3, min(K, 10))):
            flush_l2(flush)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            f()
            s1.record(stream)
            torch.cuda.synchronize()
            ts.append(s0.elapsed_time(s1))
        extra_ms[name] = float(np.median(ts))
    best = min(ms, key=ms.get)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tiling = {"fwd": rlk.det_gemm_tile_plan(rlk.RLK_GEMM_FWD, M, N, K_, sms),
              "da": rlk.det_gemm_tile_plan(rlk.RLK_GEMM_DA, M, K_, N, sms),
              "db": rlk.det_gemm_tile_plan(rlk.RLK_GEMM_DB, K_, N, M, sms)}
    line = {
        "metric": "det_gemm fwd+da+db TFLOP/s (M=N=K=4096, BF16 in/out, FP32 accumulate)",
        "value": 3 * flop * world * K / t / 1e12, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "det_gemm 4096^3 fwd+da+db, A,B~N(0,1/sqrt(K)), dC~N(0,1)",
                   "l2": "L2 flushed (256 MB write, then read) before every step"},
        "kernels_ms": ms,
        "tflops_per_op": {n: flop / (v / 1e3) / 1e12 for n, v in ms.items()},
        "roofline": {"bound": "tensor", "achieved": flop / (ms[best] / 1e3) / 1e12, "peak": peak,
                     "unit": "TFLOP/s", "frac": flop / (ms[best] / 1e3) / 1e12 / peak,
                     "traffic": measured_traffic("det_gemm_kernel", f"det_gemm 4096^3 {best}"),
                     "traffic_unit": "bytes per launch (ncu dram read+write)",
                     "kernel": f"det_gemm_kernel ({best})",
                     "algorithmic": f"2*M*N*K = {flop:.4g} FLOP per launch; "
                                    f"{2 * (M * K_ + K_ * N) + 2 * M * N} bytes (bf16 out)",
                     "peak_kind": f"{peak_src} burst bf16"},
        "cublas_bf16_tflops_context": cublas,
        "other_entry_points_ms_median": extra_ms,
        "clocks": clocks.summary(),
        "tiling": tiling,
        "gpu_launches": K * sum(p["launches"] for p in tiling.values()),
    }
    line["roofline"].update(per_clock(line["roofline"]["achieved"], line["clocks"], dev))
    # ---- e2e: host buffers (pinned) in, all three results out, copies timed.  Two
    # input / output sets alternate: a step's host-to-device copies (h2d stream)
    # and the previous step's device-to-host copies (d2h stream) overlap the
    # kernels, and every step still moves all of its bytes inside the timed region.
    if not args.no_e2e:
        Ah, Bh, dCh = (x.cpu().pin_memory() for x in (A, B, dC))
        outs_h = [[torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
                  for _ in range(2)]
        dev_in = [(A, B, dC), tuple(torch.empty_like(x) for x in (A, B, dC))]
        dev_out = [[torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(3)]
                   for _ in range(2)]
        h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        in_free, out_free = [None, None], [None, None]
        E = max(3, min(K, 10))
        lib = rlk.lib()
        P, sp = rlk._ptr, rlk._stream_ptr(None)
        for i in range(E + 2):
            b = i % 2
            a_, b_, d_ = dev_in[b]
            if i == 2:
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                h2d.wait_event(e0)
                d2h.wait_event(e0)
            if in_free[b] is not None:
                h2d.wait_event(in_free[b])
            with torch.cuda.stream(h2d):
                a_.copy_(Ah, non_blocking=True)
                b_.copy_(Bh, non_blocking=True)
                d_.copy_(dCh, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(h2d)
            stream.wait_event(ready)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])        # the d2h copies of set b are done
            o = dev_out[b]
            rlk._check(lib.rlk_det_gemm_fwd(P(a_), M, K_, K_, P(b_), N, N, P(o[0]), rlk.RLK_BF16, N,
                                            None, 0, sp), "rlk_det_gemm_fwd")
            rlk._check(lib.rlk_det_gemm_da(P(d_), rlk.RLK_BF16, M, N, N, P(b_), K_, N, P(o[1]),
                                           rlk.RLK_BF16, K_, None, 0, sp), "rlk_det_gemm_da")
            rlk._check(lib.rlk_det_gemm_db(P(a_), M, K_, K_, P(d_), rlk.RLK_BF16, N, N, P(o[2]),
                                           rlk.RLK_BF16, N, None, 0, sp), "rlk_det_gemm_db")
            in_free[b] = torch.cuda.Event()
            in_free[b].record(stream)
            d2h.wait_event(in_free[b])
            with torch.cuda.stream(d2h):
                for hst, dv in zip(outs_h[b], o):
                    hst.copy_(dv, non_blocking=True)
            out_free[b] = torch.cuda.Event()
            out_free[b].record(d2h)
        stream.wait_stream(d2h)
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        torch.cuda.synchronize()
        te = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        assert all(torch.equal(x, y) for x, y in zip(outs_h[0], outs_h[1]))
        line["e2e"] = {"value": 3 * flop * world * E / te / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": 3 * M * K_ * 2, "d2h_bytes_per_step": 3 * M * N * 2,
                       "ms_per_step": te / E * 1e3,
                       "pipelining": "inputs and outputs double-buffered; a step's copies (one stream "
                                     "each way) overlap the neighbouring steps' kernels"}
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        rows = 2 * oracle.load().max_threads()
        tf, dt, cores = oracle_gemm_tflops(A, B, dC, rows)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"{rows} output rows of each of fwd, dA and dB at 4096^3, "
                                          f"FP64, {dt:.2f} s wall"}
    return line


def ablation_bench(args, dev, rank, world, peaks, peak_src):
    """The throughput-mode ablation: the operator (V-only split) against the same
    kernels with the occupancy-driven, N-dependent split count, whole calls
    (partials + combine) timed in alternating blocks on the mid shape."""
    import deterministic_invariant_gemm_linear_gb300 as rlk
    w = si.MID
    if args.rows:
        w = si.LinearLogpWorkload(f"{w.name} (rows={args.rows})", N=args.rows, H=w.H, V=w.V,
                                  bias=w.bias, target_mode=w.target_mode)
    hidden, weight, bias, target = si.workload_inputs(w, seed=rank, device=dev)
    s_inv = rlk.vocab_split_policy(w.V)[0]
    s_tp = rlk.throughput_split_count(w.N, w.V)
    calls = {"invariant": rlk.LinearLogpCall(hidden, weight, target, bias),
             "throughput_mode": rlk.LinearLogpCall(hidden, weight, target, bias, num_splits=s_tp)}
    for c in calls.values():
        for _ in range(args.warmup):
            c()
    torch.cuda.synchronize()
    K = args.steps
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if weight.numel() * 2 < (512 << 20) else None
    ms = {k: [] for k in calls}
    barrier(world)
    with ClockSampler(dev) as clocks:
        for _ in range(3):
            for name, c in calls.items():
                if flush is None:
                    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s.record(stream)
                    for _ in range(K):
                        c()
                    e.record(stream)
                    torch.cuda.synchronize()
                    ms[name].append(s.elapsed_time(e) / K)
                else:
                    tot = 0.0
                    for _ in range(K):
                        flush_l2(flush)
                        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        s.record(stream)
                        c()
                        e.record(stream)
                        torch.cuda.synchronize()
                        tot += s.elapsed_time(e)
                    ms[name].append(tot / K)
    assert rlk.device_error() == 0
    med = {k: float(np.median(v)) for k, v in ms.items()}
    t_inv = max_over_ranks(med["invariant"] / 1e3, world, dev)
    flops = 2.0 * w.N * w.H * w.V
    achieved = flops / t_inv / 1e12
    return {
        "metric": f"linear-logp throughput-mode ablation (N={w.N},H={w.H},V={w.V}): "
                  "V-only split vs N-dependent split",
        "value": w.N * world / t_inv, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_inv * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: N={w.N} H={w.H} V={w.V}, whole calls, 3 alternating "
                               f"blocks of {K} per mode",
                   "global_batch": w.N * world, "seq_len": None, "parallelism": f"replicas x{world}",
                   "l2": "W streamed from HBM every call" if flush is None else
                         "L2 flushed (256 MB write, then read) before every call"},
        "ablation": {"invariant": {"num_splits": s_inv, "ms_per_call": med["invariant"]},
                     "throughput_mode": {"num_splits": s_tp, "ms_per_call": med["throughput_mode"]},
                     "invariant_time_over_throughput_time":
                         med["invariant"] / med["throughput_mode"],
                     "blocks_ms": ms},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                     "kernel": "whole linear-logp call (partials + combine), V-only split",
                     "peak_kind": f"{peak_src} burst bf16"},
        "clocks": clocks.summary(),
        "gpu_launches": 2 * 2 * 3 * K,
    }


def h2d_bench(args, dev, rank, world, peaks, peak_src):
    """The host link the end-to-end legs copy through: pinned host <-> device copies of
    the mid weight's size (1.245 GB), as one copy and split over 2..16 streams, timed
    with CUDA events (best of `steps` repetitions after `warmup`)."""
    nbytes = 151936 * 4096 * 2
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    host.fill_(1)
    devbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    res = {}

    def timed(fn, streams):
        best = float("inf")
        main = torch.cuda.current_stream()
        for i in range(args.warmup + args.steps):
            torch.cuda.synchronize()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(main)
            for st in streams:
                st.wait_event(s)
            fn()
            for st in streams:
                main.wait_stream(st)
            e.record(main)
            torch.cuda.synchronize()
            if i >= args.warmup:
                best = min(best, s.elapsed_time(e) / 1e3)
        return nbytes / best / 1e9

    with ClockSampler(dev) as clocks:
        for name, direction in (("h2d", 0), ("d2h", 1)):
            for n in (1, 2, 4, 8, 16):
                streams = [torch.cuda.Stream(device=dev) for _ in range(n)]
                chunk = -(-nbytes // n)

                def run():
                    for k, st in enumerate(streams):
                        lo, hi = k * chunk, min(nbytes, (k + 1) * chunk)
                        with torch.cuda.stream(st):
                            if direction == 0:
                                devbuf[lo:hi].copy_(host[lo:hi], non_blocking=True)
                            else:
                                host[lo:hi].copy_(devbuf[lo:hi], non_blocking=True)
                res[f"{name}_{n}_streams_gbs"] = timed(run, streams)
    best_h2d = max(v for k, v in res.items() if k.startswith("h2d"))
    return {
        "metric": "pinned host-to-device copy GB/s (1.245 GB, the mid weight's size)",
        "value": best_h2d, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": nbytes / best_h2d / 1e6, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "host link: one pinned 1.245 GB buffer copied whole or split over "
                               "2-16 streams, each direction; best of steps after warmup"},
        "copies": res, "clocks": clocks.summary(), "gpu_launches": 0,
    }


def shards_bench(args, dev, rank, world, peaks, peak_src):
    """The vocabulary-parallel path on one GPU: the mid workload's vocabulary cut into
    --shards balanced runs of whole splits, each shard's partials computed from its
    own weight rows (one launch per shard, back to back), then the fixed-order merge
    over the gathered partials; against the one-call operator on the same inputs.
    The exchange between GPUs (an all-gather of N*S*8 + 4*N bytes per rank) has no
    second GPU to go to here and is not timed."""
    import deterministic_invariant_gemm_linear_gb300 as rlk
    w = si.MID
    R = args.shards
    hidden, weight, bias, target = si.workload_inputs(w, seed=rank, device=dev)
    S = rlk.vocab_split_policy(w.V)[0]
    ranges = [rlk.vocab_shard_range(w.V, R, q) for q in range(R)]
    widest = max(r[1] - r[0] for r in ranges)
    shards = [weight[v0:v1].contiguous() for _, _, v0, v1 in ranges]
    offsets = [r[0] for r in ranges] + [S]
    lib, P, sp = rlk.lib(), rlk._ptr, rlk._stream_ptr(None)
    N, H, V = w.N, w.H, w.V
    parts = torch.empty(R, N, widest, 2, dtype=torch.float32, device=dev)
    zts = torch.full((R, N), float("nan"), dtype=torch.float32, device=dev)
    wss = []
    for (j0, j1, v0, v1), ws_ in zip(ranges, shards):
        n = lib.rlk_linear_logp_shard_workspace_size(P(hidden), N, H, H, P(ws_), V, j0, j1, H)
        wss.append(torch.empty(n, dtype=torch.uint8, device=dev))
    logp = torch.empty(N, device=dev)
    lse = torch.empty(N, device=dev)
    offs = (ctypes.c_int64 * (R + 1))(*offsets)

    def shard(q):
        j0, j1, v0, v1 = ranges[q]
        rlk._check(lib.rlk_linear_logp_shard_partials(
            P(hidden), N, H, H, P(shards[q]), V, j0, j1, H, None, P(target), 1, P(parts[q]), widest,
            P(zts[q]), P(wss[q]), wss[q].numel(), sp), "rlk_linear_logp_shard_partials")

    def merge():
        rlk._check(lib.rlk_linear_logp_combine_shards(
            N, V, P(target), 1, R, offs, P(parts), widest, N * widest, P(zts), N, P(logp), P(lse),
            None, sp), "rlk_linear_logp_combine_shards")

    one = rlk.LinearLogpCall(hidden, weight, target, bias)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for q in range(R):
            shard(q)
        merge()
        one()
    torch.cuda.synchronize()
    assert torch.equal(logp, one.logp) and torch.equal(lse, one.lse), "shards must equal one call"
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(R + 2)] for _ in range(K)]
    barrier(world)
    with ClockSampler(dev) as clocks:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(K):
            ev[k][0].record(stream)
            for q in range(R):
                shard(q)
                ev[k][q + 1].record(stream)
            merge()
            ev[k][R + 1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    t = max_over_ranks(start.elapsed_time(end) / 1e3, world, dev)
    shard_ms = [float(np.mean([e[q].elapsed_time(e[q + 1]) for e in ev])) for q in range(R)]
    merge_ms = float(np.mean([e[R].elapsed_time(e[R + 1]) for e in ev]))
    o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    o0.record(stream)
    for _ in range(K):
        one()
    o1.record(stream)
    torch.cuda.synchronize()
    one_ms = o0.elapsed_time(o1) / K
    assert rlk.device_error() == 0
    flops = 2.0 * N * H * V
    q_big = max(range(R), key=lambda q: ranges[q][3] - ranges[q][2])
    vq = ranges[q_big][3] - ranges[q_big][2]
    achieved = 2.0 * N * H * vq / (shard_ms[q_big] / 1e3) / 1e12
    line = {
        "metric": f"vocabulary-parallel linear-logp on one GPU ({R} shards back to back + merge; "
                  f"N={N},H={H},V={V})",
        "value": N * world * K / t, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: N={N} H={H} V={V}, {R} balanced shards of whole splits",
                   "shards": [{"splits": [j0, j1], "ids": [v0, v1]} for j0, j1, v0, v1 in ranges],
                   "l2": f"inputs larger than L2: W {V * H * 2 / 1e9:.3f} GB streamed per step"},
        "kernels_ms": {"shard_partials": shard_ms, "combine_shards": merge_ms},
        "one_call_ms": one_ms,
        "shards_over_one_call": (sum(shard_ms) + merge_ms) / one_ms,
        "bitwise_equal_to_one_call": True,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                     "kernel": f"linear_logp_partials_kernel on shard {q_big} ({vq} ids)",
                     "algorithmic": f"2*N*H*V_shard = {2.0 * N * H * vq:.4g} FLOP per launch",
                     "peak_kind": f"{peak_src} burst bf16"},
        "exchange": f"not timed (one GPU): {N * S * 8 + 4 * N} bytes gathered per step in total",
        "clocks": clocks.summary(),
        "gpu_launches": (R + 1) * K,
    }
    line["roofline"].update(per_clock(achieved, line["clocks"], dev))
    return line


def secondary_measurements(dev, peaks, steps: int = 10):
    """Compact measurements of the other workloads, carried by the default line so that
    they are recorded in the same run: partials kernel times (CUDA events on the
    launching stream, L2 flushed before each launch when the weight fits in it) for
    ragged N=17 / 255 and the large workload, the whole tiny call, det_gemm fwd / dA /
    dB at 4096^3 (L2 flushed) and the mid backward step."""
    import deterministic_invariant_gemm_linear_gb300 as rlk
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}

    def timed(fn, cold):
        ts = []
        with ClockSampler(dev) as clocks:
            for i in range(3 + steps):
                if cold:
                    flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize()
                if i >= 3:
                    ts.append(e0.elapsed_time(e1))
        sm = (clocks.summary() or {}).get("sm_mhz")
        return float(np.median(ts)), float(np.min(ts)), sm

    for name, w in (("ragged_N17", si.ragged(17)), ("ragged_N255", si.ragged(255)), ("large", si.LARGE),
                    ("tiny", si.TINY)):
        hidden, weight, bias, target = si.workload_inputs(w, seed=0, device=dev)
        call = rlk.LinearLogpCall(hidden, weight, target, bias)
        cold = weight.numel() * 2 < (512 << 20)
        med, best, mhz = timed(call if name == "tiny" else call.partials, cold)
        S = rlk.vocab_split_policy(w.V)[0]
        alg = 2 * w.V * w.H + 2 * w.N * w.H + 8 * w.N + 8 * w.N * S + 4 * w.N + (4 * w.V if w.bias else 0)
        flops = 2.0 * w.N * w.H * w.V
        rec = {"what": ("whole call" if name == "tiny" else "partials kernel") +
                       (", L2 flushed (write + read) before each" if cold else ", W streamed from HBM"),
               "ms_median": med, "ms_best": best, "sm_mhz": mhz}
        if name.startswith("ragged"):
            rec["hbm_frac"] = alg / (med / 1e3) / 1e9 / peaks["hbm_gbs"]
        elif name == "large":
            rec["bf16_frac"] = flops / (med / 1e3) / 1e12 / peaks["bf16_tflops"]
        out[name] = rec
        del hidden, weight, bias, target, call
    A, B, dC = si.det_gemm_inputs(4096, 4096, 4096, seed=0, device=dev)
    flop = 2.0 * 4096 ** 3
    dg = {}
    for op, fn in (("fwd", lambda: rlk.det_gemm_fwd(A, B)), ("da", lambda: rlk.det_gemm_da(dC, B)),
                   ("db", lambda: rlk.det_gemm_db(A, dC))):
        med, best, mhz = timed(fn, True)
        dg[op] = {"ms_median": med, "ms_best": best, "sm_mhz": mhz,
                  "bf16_frac": flop / (med / 1e3) / 1e12 / peaks["bf16_tflops"]}
    out["det_gemm_4096"] = dg
    del A, B, dC
    w = si.MID
    hidden, weight, bias, target = si.workload_inputs(w, seed=0, device=dev)
    g = torch.randn(w.N, device=dev, generator=torch.Generator(device=dev).manual_seed(7))
    _, lse = rlk.linear_logp(hidden, weight, target, bias)
    med, best, mhz = timed(lambda: rlk.linear_logp_backward(hidden, weight, target, lse, g,
                                                       out_dtype=torch.bfloat16), False)
    out["backward_mid"] = {"ms_median": med, "ms_best": best, "sm_mhz": mhz,
                           "bf16_frac": 3 * 2.0 * w.N * w.H * w.V / (med / 1e3) / 1e12 /
                           peaks["bf16_tflops"],
                           "what": "whole backward call (G kernel + grad_hidden + grad_weight, "
                                   "outputs allocated by the binding)"}
    assert rlk.device_error() == 0
    return out


def reference_arm(args):
    """The FP64 CPU oracle as the reference implementation, on a bounded sample.

    Each step runs the oracle on `cores` rows (one per host thread) against a
    contiguous slice of Vs vocabulary rows, Vs sized so that warm-up + steps end
    within about 150 s; the oracle's cost is linear in V, so its throughput is
    reported in full-vocabulary rows per second (rows * Vs / V per step).
    """
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    orc = oracle.load()
    w = {"mid": si.MID, "large": si.LARGE}.get(args.workload, si.MID)
    cores = orc.max_threads()
    g = torch.Generator().manual_seed(0)
    hidden = torch.randn(cores, w.H, generator=g).to(torch.bfloat16)
    weight = (torch.randn(w.V, w.H, generator=g) / math.sqrt(w.H)).to(torch.bfloat16)
    target = torch.randint(0, w.V, (cores,), generator=g)
    bias = (torch.randn(w.V, generator=g) * 0.01) if w.bias else None
    hb, wb, tb = si.bf16_bits(hidden), si.bf16_bits(weight), target.numpy()
    bb = None if bias is None else bias.numpy()
    t0 = time.perf_counter()
    orc.linear_logp(hb[:1], wb, tb[:1], bb, threads=1)          # one full row, one thread
    t_row = time.perf_counter() - t0
    step_budget = 150.0 / (args.steps + args.warmup)
    Vs = max(256, min(w.V, int(w.V * step_budget / max(t_row, 1e-9))))
    ws, tsb = wb[:Vs], tb % Vs
    bs = None if bb is None else bb[:Vs]
    for _ in range(args.warmup):
        orc.linear_logp(hb, ws, tsb, bs, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.linear_logp(hb, ws, tsb, bs, threads=cores)
    dt = time.perf_counter() - t0
    value = cores * (Vs / w.V) * args.steps / dt
    sample = (f"{cores} rows x {Vs} of {w.V} vocabulary rows per step of the {w.name} workload "
              f"(full H); reported as full-vocabulary rows/s")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {
        "impl": "reference", "metric": linear_logp_metric(w),
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": linear_logp_config(w, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mid",
                    choices=["mid", "large", "tiny", "ragged", "det_gemm", "backward", "ablation", "h2d",
                             "shards"])
    ap.add_argument("--impl", default="rlk", choices=["rlk", "reference"])
    ap.add_argument("--rows", type=int, default=0,
                    help="override the row count N of a linear-logp workload (profiling cases)")
    ap.add_argument("--shards", type=int, default=2, help="--workload shards: number of shards")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-secondary", action="store_true",
                    help="default workload: skip the compact measurements of the other workloads")
    ap.add_argument("--phases", action="store_true",
                    help="linear-logp: per-phase breakdown of the partials kernel from the debug "
                         "build's trace (needs RLK_LIBRARY=debug)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        line = reference_arm(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, src = load_peaks()
    if args.workload == "det_gemm":
        line = det_gemm_bench(args, dev, rank, world, peaks, src)
    elif args.workload == "backward":
        line = backward_bench(args, dev, rank, world, peaks, src)
    elif args.workload == "ablation":
        line = ablation_bench(args, dev, rank, world, peaks, src)
    elif args.workload == "h2d":
        line = h2d_bench(args, dev, rank, world, peaks, src)
    elif args.workload == "shards":
        line = shards_bench(args, dev, rank, world, peaks, src)
    else:
        line = linear_logp_bench(args, dev, rank, world, peaks, src)
        if (args.workload == "mid" and not args.rows and not args.no_secondary and world == 1
                and not args.phases):
            line["secondary"] = secondary_measurements(dev, peaks)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
