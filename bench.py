#!/usr/bin/env python3
"""Throughput of the NVFP4 quantizer's hot path on one GB300 (or N replicas).

A step is one pass of the whole path over one batch: the global amax pass and
the fused quantize (RHT + Philox stochastic rounding + E4M3/E2M1 encode +
packing + 32x4x4-swizzled scales) over an 8192x4096 bf16 activation with 0.1%
outlier columns.  The metric is effective HBM GB/s: bf16 bytes read (the amax
pass included) plus codes, scales and the scale words written, divided by the
step time.  Inputs are resident in HBM before the timed region and the L2 is
flushed before every timed step (a 512 MiB write, then a 256 MiB read of
another buffer, so the cache starts cold and holds no dirty lines).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores (the pages publish no runnable implementation).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tensor_quantization_gb300 import workloads as wl  # noqa: E402

METRIC = "NVFP4 quantize effective HBM GB/s and % of GB300 peak (8192×4096 bf16, RHT+SR)"
UNIT = "GB/s"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- bytes
def scale_bytes(rows_out: int, cols_out: int, swizzled: bool) -> int:
    cs = cols_out // 16
    if not swizzled:
        return rows_out * cs
    return ((rows_out + 127) // 128 * 128) * ((cs + 3) // 4 * 4)


def orientations(w: wl.Workload):
    out = []
    if w.rowwise:
        out.append((w.rows, w.cols))
    if w.colwise:
        out.append((w.cols, w.rows))
    return out


def two_scales(w: wl.Workload) -> bool:
    """RHT in both orientations: one amax and global scale per orientation."""
    return w.rht and w.rowwise and w.colwise and not w.amax_given


def counted_bytes(w: wl.Workload, elem: int = 2) -> dict:
    """Algorithmic bytes of one step.  Per tensor: the amax pass reads the input
    and writes amax and g (8 B); the encode reads it again and writes codes and
    scales.  Per row: one read serves both, plus 8 B of scale words per row."""
    n = w.rows * w.cols
    codes = sum(r * c // 2 for r, c in orientations(w))
    scales = sum(scale_bytes(r, c, w.swizzled) for r, c in orientations(w))
    if w.amax_given:  # one read; the given amax is read and g written
        q = n * elem + codes + scales + 8
        return {"amax_pass": 0, "quantize": q, "total": q}
    if w.groups:  # amax pass and encode each read the input once; amax and g per group
        ng = len(w.groups) - 1
        a, q = n * elem + 8 * ng, n * elem + codes + scales
        return {"amax_pass": a, "quantize": q, "total": a + q}
    if two_scales(w):  # one amax read serves both orientations, with two amax/g pairs
        a, q = n * elem + 16, n * elem + codes + scales
        return {"amax_pass": a, "quantize": q, "total": a + q}
    if w.per_row:
        q = n * elem + codes + scales + 8 * w.rows
        return {"amax_pass": 0, "quantize": q, "total": q}
    a, q = n * elem + 8, n * elem + codes + scales
    return {"amax_pass": a, "quantize": q, "total": a + q}


# ---------------------------------------------------------------- peaks
def clk_max_mhz() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["sm_max_mhz"])
    except Exception:
        return 2070.0


def hbm_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_field(kernel: str, workload: str, field: str) -> float | None:
    """A number recorded in the committed ncu summary of this kernel on this
    workload (profiles/<kernel>__<workload>.md), if the summary's source digest
    matches the current kernel sources; None otherwise."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(field + r":\s*([0-9.eE+]+)", text)
    s = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_digest():
        return None
    return float(m.group(1))


def choose_roofline(w: wl.Workload, hbm_view: dict, issue_view: dict | None, traffic) -> dict:
    """The roofline a workload is judged against: plain ALU issue for the
    per-row four-over-six path (two candidates per block), with its HBM view
    beside it; HBM bandwidth of the counted bytes for the codec workloads, with
    the issue rate the kernel runs at beside it (when ncu's count is known)."""
    if issue_view is None:
        return hbm_view
    if w.per_row:
        return dict(issue_view, traffic=traffic, hbm_view={k: hbm_view[k] for k in ("achieved", "peak", "unit", "frac")})
    return dict(hbm_view, issue_view={k: issue_view[k] for k in ("achieved", "peak", "unit", "frac", "peak_source")})


def profile_traffic(kernel: str, workload: str) -> float | None:
    return profile_field(kernel, workload, "traffic_bytes_per_launch")


# Host-only entry-point files (argument checks and the choice of launches):
# no kernel code or launch configuration, so not part of the kernel digest.
HOST_ONLY_SOURCES = ("nvfp4_api.cu", "nvfp4_static.cu")


def source_digest() -> str:
    """Digest of the kernel sources (device code and its launchers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_quantization_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in HOST_ONLY_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read only) on a
    background thread while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period, self._stop = period_s, threading.Event()
        self.ok = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.nv, self.h, self.ok = nv, h, True
        except OSError:
            pass

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self) -> dict:
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self.ok else "unavailable"}


# ------------------------------------------------------------ ranks
def max_over_ranks(value: float, world: int, device) -> float:
    """The slowest rank's timed total: every rank's number, MAX-reduced."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step: int, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank processes its own batch (replicas),
    all in the slowest rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------- our arm
def bench_config(w: wl.Workload, world: int) -> dict:
    """The workload description both arms report."""
    return {"workload": w.name, "rows": w.rows, "cols": w.cols, "input": "bf16", "mode": w.mode, "rht": w.rht,
            "amax": "given (NVFP4_AMAX_GIVEN, computed before the timed region)" if w.amax_given else "computed",
            "scales": "swizzled_32x4x4" if w.swizzled else "linear",
            "l2": "flushed before every timed step: 512 MiB write + 256 MiB read",
            "parallelism": f"replicas{world}" if world > 1 else "single_gpu"}


def run_ours(args, rank: int, world: int) -> dict | None:
    from tensor_quantization_gb300 import build, nvfp4

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    nvfp4.load()
    w = workload_of(args)
    x_cpu, mask = wl.make_input(w)
    x = x_cpu.to(dev)
    R, C = w.rows, w.cols
    flags = (nvfp4.ROWWISE if w.rowwise else 0) | (nvfp4.COLWISE if w.colwise else 0) | \
        (nvfp4.SWIZZLED if w.swizzled else 0) | (nvfp4.BLOCK_2D if w.block2d else 0) | \
        (nvfp4.SCALE_PER_ROW if w.per_row else 0)
    q = nvfp4.alloc_outputs(x, flags, w.rht)  # two amax / global scale slots for RHT in both orientations
    if w.groups:  # one amax / global scale per group
        offs_d = torch.tensor(w.groups, dtype=torch.int64, device=dev)
        q = nvfp4.Quantized(q.codes_row, q.scales_row, None, None,
                            torch.empty(len(w.groups) - 1, dtype=torch.float32, device=dev),
                            torch.empty(len(w.groups) - 1, dtype=torch.float32, device=dev), flags)
    out = nvfp4.make_output(q.codes_row, q.scales_row, q.codes_col, q.scales_col, q.amax, q.global_scale)
    ws = nvfp4.Workspace.get(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scrub = torch.ones(L2_FLUSH_BYTES // 2, dtype=torch.uint8, device=dev)

    def flush_l2(k: int) -> None:
        flush.fill_(k & 0xFF)  # evicts everything
        scrub.max()  # write-back of the dirty flush lines happens here, untimed
    amax_kernel, quant_kernel = kernel_plan(w)
    # the split loop's amax pass is the standalone entry point, whose kernel
    # differs from the call's with the RHT
    split_amax = ("k_amax_rht_col" if w.colwise else "k_amax_ldg_rht") if w.rht else amax_kernel
    # two kernels: amax pass then encode, also timed separately (a two-scale
    # call runs four kernels and is timed as one call)
    split = amax_kernel is not None and not multi_kernel_call(w)
    orient_flag = nvfp4.COLWISE if (w.colwise and not w.rowwise) else nvfp4.ROWWISE
    if w.amax_given:  # the amax a caller would bring (e.g. from delayed scaling), outside the timed region
        nvfp4.nvfp4_amax(x, orient_flag, w.rht, mask, out, ws, stream)
        torch.cuda.synchronize(dev)
        flags |= nvfp4.AMAX_GIVEN

    def quant_call(fl):
        if w.groups:
            mode = {"rne": nvfp4.MODE_RNE, "4o6": nvfp4.MODE_FOUR_OVER_SIX}.get(
                w.mode, nvfp4.MODE_RHT_SR if w.rht else nvfp4.MODE_SR)
            nvfp4.nvfp4_quantize_grouped(x, fl, offs_d, len(w.groups) - 1, mode, mask, w.philox_seed,
                                         w.philox_offset, out, stream)
        elif w.mode == "sr" and w.rht:
            nvfp4.nvfp4_quantize_rht_sr(x, fl, mask, w.philox_seed, w.philox_offset, out, ws, stream)
        elif w.mode == "sr":
            nvfp4.nvfp4_quantize_sr(x, fl, w.philox_seed, w.philox_offset, out, ws, stream)
        elif w.mode == "4o6":
            nvfp4.nvfp4_quantize_four_over_six(x, fl, out, ws, stream)
        else:
            nvfp4.nvfp4_quantize_rne(x, fl, out, ws, stream)

    def step(ev0, ev1, ev2):
        ev0.record(stream)
        if split:
            nvfp4.nvfp4_amax(x, orient_flag, w.rht, mask, out, ws, stream)
            ev1.record(stream)
            quant_call(flags | nvfp4.AMAX_GIVEN)
        else:
            ev1.record(stream)
            quant_call(flags)
        ev2.record(stream)

    def fused_step(ev0, ev1):
        ev0.record(stream)
        quant_call(flags)  # the public call: amax pass + quantize pass
        ev1.record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        flush_l2(1)
        fused_step(*[torch.cuda.Event(enable_timing=True) for _ in range(2)])
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for k in range(args.steps):
            flush_l2(k)
            fused_step(*evs[k])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), world, dev)

    # per-kernel durations: the same steps issued as two calls with an event
    # between the passes (same kernels; the event keeps them from overlapping).
    # A one-kernel call is its own kernel duration.
    if split:
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for k in range(args.steps):
            flush_l2(k)
            step(*sevs[k])
        torch.cuda.synchronize(dev)
        k1_ms = [e[0].elapsed_time(e[1]) for e in sevs]
        k2_ms = [e[1].elapsed_time(e[2]) for e in sevs]
        split_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in sevs)
    else:
        k1_ms, k2_ms = [0.0], step_ms
        split_ms = statistics.mean(step_ms)

    # end to end through the public API: pinned host input -> device, the
    # fused call (amax pass + encode), codes/scales/scale words -> pinned host
    x_host = x_cpu.pin_memory()
    host_out = {k: torch.empty(getattr(q, k).shape, dtype=getattr(q, k).dtype, pin_memory=True)
                for k in ("codes_row", "scales_row", "codes_col", "scales_col", "amax", "global_scale")
                if getattr(q, k) is not None}
    e2e_ms = []
    for k in range(max(3, min(args.steps, 20)) + 2):
        flush_l2(7)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x.copy_(x_host, non_blocking=True)
        quant_call(flags)
        for name, h in host_out.items():
            h.copy_(getattr(q, name), non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        if k >= 2:
            e2e_ms.append(a.elapsed_time(b))
    h2d = x_cpu.numel() * x_cpu.element_size()
    d2h = sum(h.numel() * h.element_size() for h in host_out.values())

    nbytes = counted_bytes(w)
    ms = total_ms / args.steps
    value = aggregate_gbs(nbytes["total"], ms, world)
    peak, peak_src = hbm_peak()
    k1, k2 = statistics.mean(k1_ms), statistics.mean(k2_ms)
    if split and k1 > k2:
        dom, dom_bytes, dom_ms, unit_desc = split_amax, nbytes["amax_pass"], k1, "2 B read per element"
    elif split:
        dom, dom_bytes, dom_ms = quant_kernel, nbytes["quantize"], k2
        unit_desc = "2 B read + 0.5 B codes + 1/16 B scale per element (+ scale words)"
    elif two_scales(w):
        dom, dom_bytes, dom_ms = "call", nbytes["total"], k2
        unit_desc = "2 B read twice (amax, encode) + 2 x (0.5 B codes + 1/16 B scale) per element"
    elif w.groups:
        dom, dom_bytes, dom_ms = "call", nbytes["total"], k2
        unit_desc = "2 B read twice (group amaxes, encode) + 0.5 B codes + 1/16 B scale per element"
    else:
        dom, dom_bytes, dom_ms = quant_kernel, nbytes["total"], k2
        unit_desc = ("2 B read + 0.5 B codes + 1/16 B scale per element + 8 B of scale words per row" if w.per_row
                     else "2 B read + 0.5 B codes + 1/16 B scale per element (amax given)" if w.amax_given
                     else "2 B read twice (amax pass, encode) + 0.5 B codes + 1/16 B scale per element")
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = profile_traffic(dom, w.name)
    hbm_view = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s", "algorithmic_bytes_per_launch": dom_bytes,
                "per_unit": unit_desc, "ms_per_launch": round(dom_ms, 5)}
    roofline = hbm_view
    wipe = profile_field(dom, w.name, "warp_inst_per_element")
    if wipe:
        # the achieved instruction rate from ncu's instruction count, against 1
        # warp instruction per cycle per scheduler: the encode kernels read
        # their input from L2 and are issue-bound
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clk_max_mhz()
        inst = wipe * R * C
        peak_i = sms * 4 * mhz * 1e6 / 1e9
        ach_i = inst / (dom_ms * 1e-3) / 1e9
        issue_view = {"bound": "alu", "kernel": dom, "achieved": round(ach_i, 1), "peak": round(peak_i, 1),
                      "unit": "Gwarp-inst/s", "frac": round(ach_i / peak_i, 4),
                      "peak_source": f"{sms} SMs x 4 schedulers x 1 warp-instruction/cycle x {mhz:.0f} MHz max SM clock",
                      "instructions_per_launch": round(inst),
                      "instructions_source": f"ncu smsp__inst_executed.sum per element, profiles/{dom}__{w.name}.md",
                      "ms_per_launch": round(dom_ms, 5)}
        roofline = choose_roofline(w, hbm_view, issue_view, traffic)
    med = statistics.median(step_ms)
    cfg = bench_config(w, world)
    cfg["input_sha256"] = hashlib.sha256(x_cpu.contiguous().view(torch.int16).numpy().tobytes()).hexdigest()
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": cfg,
        # this rank's median step beside the mean (CUDA event ticks are ~2 us apart on this GPU: the mean
        # over many steps resolves finer than any single step)
        "ms_per_step_median": round(med, 5), "value_median": round(aggregate_gbs(nbytes["total"], med, world), 1),
        "torch": torch.__version__,
        "counted_bytes_per_step": nbytes["total"],
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": roofline,
        "kernels_ms": ({split_amax: round(k1, 5), quant_kernel: round(k2, 5), "split_step": round(split_ms, 5),
                        "source": "second loop: the standalone amax pass, an event, the encode with the amax given"}
                       if split else
                       {"call": round(k2, 5), "source": f"the timed steps ({len(call_kernels(w))} kernels per call)"}
                       if multi_kernel_call(w) else
                       {quant_kernel: round(k2, 5), "source": "the timed steps (one kernel per call)"}),
        "e2e": {"value": round(nbytes["total"] / (statistics.mean(e2e_ms) * 1e-3) / 1e9, 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(statistics.mean(e2e_ms), 4)},
        "gpu_launches": args.steps * len(call_kernels(w)) + (args.steps if pad_launch_needed(w) else 0),
        "kernels": call_kernels(w),
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    return res


def workload_of(args) -> wl.Workload:
    w = wl.WORKLOADS[args.workload]
    if args.shape:
        r, c = (int(v) for v in args.shape.lower().split("x"))
        w = w.resized(r, c)
    return w


FUSED_MAX_ELEMS = 1 << 22  # the library's one-kernel limit for per-tensor rowwise calls
ROWSCALED_STAGED_MAX_ROW_BYTES = 96 * 1024


def kernel_plan(w: wl.Workload) -> tuple[str | None, str]:
    """(amax kernel or None, quantize kernel) that one call of this workload
    launches, by the library's dispatch rules."""
    if w.per_row:
        return None, ("k_quant_rowscaled_staged" if w.cols * 2 <= ROWSCALED_STAGED_MAX_ROW_BYTES
                      else "k_quant_rowscaled")
    if w.groups:
        return "k_amax_groups", "k_quant_row_grouped"
    if w.amax_given:  # the quantize kernel alone (the one-kernel path needs to compute the amax)
        return None, ("k_quant_2d" if w.block2d else "k_quant_col" if not w.rowwise else "k_quant_row")
    if w.rowwise and not w.colwise and not w.block2d and w.rows * w.cols <= FUSED_MAX_ELEMS:
        return None, "k_quant_row_fused"
    # bf16 RHT column blocks (alone, or with the row blocks of the same read);
    # RHT row blocks of a contiguous bf16 input: the load-based pass
    amax = "k_amax_tma_cols" if (w.rht and w.colwise) else "k_amax_ldg_rht" if w.rht else "k_amax_tma"
    if w.block2d:
        return amax, "k_quant_2d"
    if w.colwise and not w.rowwise:
        return amax, "k_quant_col"
    return amax, "k_quant_row"


def call_kernels(w: wl.Workload) -> list[str]:
    """Every kernel one call of this workload launches (the scale pad aside)."""
    if two_scales(w):  # one amax read for both orientations
        return ["k_amax_tma_cols", "k_quant_row", "k_quant_col"]
    if w.groups:
        return ["k_amax_groups", "k_group_finalize", "k_quant_row_grouped"]
    return [k for k in kernel_plan(w) if k]


def multi_kernel_call(w: wl.Workload) -> bool:
    """Calls that launch more than an amax pass and one encode: timed as one call."""
    return two_scales(w) or bool(w.groups)


def pad_launch_needed(w: wl.Workload) -> bool:
    if not w.swizzled:
        return False
    for r, c in orientations(w):
        if r % 128 or (c // 16) % 4:
            return True
    return False


# ------------------------------------------------------------ the oracle
def oracle_sample(w: wl.Workload, x_cpu: torch.Tensor, mask: int, rows: int, amax: float | None = None,
                  threads: int = 1):
    """One oracle pass (amax + encode; the encode alone with a given amax)
    over the first `rows` rows, single-threaded or over `threads` host threads
    (row ranges; the same result bit for bit)."""
    import numpy as np

    import oracle
    xs = x_cpu[:rows].contiguous().view(torch.int16).numpy().view(np.uint16)
    par = threads > 1
    if w.groups:  # each group (clipped to the sample) is its own tensor: amax, then encode
        for o0, o1 in zip(w.groups[:-1], w.groups[1:]):
            o1 = min(o1, rows)
            if o0 >= o1:
                continue
            kw = dict(mode=w.mode, swizzled=w.swizzled, rht=w.rht, sign_mask=mask, seed=w.philox_seed,
                      offset=w.philox_offset, row_range=(o0, o1))
            if par:
                A = oracle.amax_parallel(xs[o0:o1], rht=w.rht, sign_mask=mask, threads=threads)
                oracle.quantize_parallel(xs, threads=threads, amax_given=A, **kw)
            else:
                A, _ = oracle.amax(xs[o0:o1], rht=w.rht, sign_mask=mask)
                oracle.quantize(xs, amax_given=float(A[0]), **kw)
        return
    for colwise in ([False] if w.rowwise else []) + ([True] if w.colwise else []):
        kw = dict(colwise=colwise, mode=w.mode, block2d=w.block2d, per_row=w.per_row, swizzled=w.swizzled,
                  rht=w.rht, sign_mask=mask, seed=w.philox_seed, offset=w.philox_offset, amax_given=amax)
        if par:
            oracle.quantize_parallel(xs, threads=threads, **kw)
        else:
            oracle.quantize(xs, **kw)


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the baseline's record."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def given_amax(w: wl.Workload, x_cpu: torch.Tensor, mask: int) -> float | None:
    """The amax a given-amax workload's calls receive (the oracle's), else None."""
    if not w.amax_given:
        return None
    import numpy as np

    import oracle
    xs = x_cpu.contiguous().view(torch.int16).numpy().view(np.uint16)
    return float(oracle.amax(xs, colwise=w.colwise and not w.rowwise, rht=w.rht, sign_mask=mask)[0][0])


def timed_passes(w, x_cpu, mask, A, threads, min_seconds):
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_sample(w, x_cpu, mask, w.rows, A, threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return reps, el


def cpu_baseline(w: wl.Workload, x_cpu: torch.Tensor, mask: int, min_seconds: float) -> dict:
    """The oracle as it stands on the host: over all host cores (row ranges on
    threads, bit-identical to one thread), and single-threaded beside it."""
    import oracle
    oracle.build()
    A = given_amax(w, x_cpu, mask)
    n = oracle.host_threads()
    reps, el = timed_passes(w, x_cpu, mask, A, n, min_seconds / 2)
    reps1, el1 = timed_passes(w, x_cpu, mask, A, 1, min_seconds / 2)
    total = counted_bytes(w)["total"]
    return {"value": round(reps * total / el / 1e9, 4), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{reps} full pass(es) of the {w.rows}x{w.cols} workload, C oracle on {n} host threads "
                      f"(row ranges), {el:.1f} s",
            "single_thread": {"value": round(reps1 * total / el1 / 1e9, 4), "cores": 1,
                              "sample": f"{reps1} full pass(es), one thread, {el1:.1f} s"},
            "nproc": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args) -> dict:
    import oracle
    oracle.build()
    w = wl.WORKLOADS[args.workload]
    x_cpu, mask = wl.make_input(w)
    rows = min(w.rows, 4096)  # a bounded sample: the first rows of the workload
    sub = wl.Workload(**{**w.__dict__, "rows": rows})
    A = given_amax(w, x_cpu, mask)
    n = oracle.host_threads()
    for _ in range(args.warmup):
        oracle_sample(w, x_cpu, mask, rows, A, n)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample(w, x_cpu, mask, rows, A, n)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    v = counted_bytes(sub)["total"] / (ms * 1e-3) / 1e9
    sample = (f"rows 0..{rows} of the {w.rows}x{w.cols} workload per step (amax + encode), C oracle on {n} host "
              f"threads (row ranges)")
    return {"metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
            "config": bench_config(w, 1),
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------- the read-bandwidth bound
READ_PROBE_SRC = r"""
#include <cstdint>
#include <cuda_runtime.h>
// every thread keeps U 16-byte loads in flight; the maximum of an xor of each
// word keeps the loads live; one atomicMax per warp
template <int U>
__global__ void read_max(const uint4 *p, long long n, unsigned *out) {
    unsigned m = 0;
    long long i = (long long)blockIdx.x * blockDim.x * U + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x * U;
    for (; i + (long long)(U - 1) * blockDim.x < n; i += stride) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; u++)
            asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w) : "l"(p + i + u * blockDim.x));
#pragma unroll
        for (int u = 0; u < U; u++) m = max(m, v[u].x ^ v[u].y ^ v[u].z ^ v[u].w);
    }
    for (; i < n; i += blockDim.x) { uint4 v = p[i]; m = max(m, v.x ^ v.y ^ v.z ^ v.w); }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}
extern "C" int read_probe(const void *p, long long bytes, unsigned *out, int ctas_per_sm, int in_flight,
                          void *stream) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaStream_t s = (cudaStream_t)stream;
    if (in_flight == 8) read_max<8><<<sms * ctas_per_sm, 256, 0, s>>>((const uint4 *)p, bytes / 16, out);
    else read_max<4><<<sms * ctas_per_sm, 256, 0, s>>>((const uint4 *)p, bytes / 16, out);
    return (int)cudaGetLastError();
}
"""


def read_sweep(args) -> dict:
    """Event time of a plain read of N MiB right after the bench's L2 flush (the
    bound of any pass that must read the input from HBM), beside the library's
    standalone amax passes on the headline input."""
    import subprocess
    import tempfile

    from tensor_quantization_gb300 import build, nvfp4
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    nvfp4.load()
    tmp = tempfile.mkdtemp()
    with open(os.path.join(tmp, "read_probe.cu"), "w") as f:
        f.write(READ_PROBE_SRC)
    so = os.path.join(tmp, "libread_probe.so")
    subprocess.run([build.nvcc(), *build.ARCH, "-O3", "-Xcompiler", "-fPIC", "-shared",
                    os.path.join(tmp, "read_probe.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.read_probe.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                               ctypes.c_void_p]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scrub = torch.ones(L2_FLUSH_BYTES // 2, dtype=torch.uint8, device=dev)
    buf = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def timed(call, reps):
        ts = []
        for k in range(reps + 3):
            flush.fill_(k & 0xFF)
            scrub.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            e1.synchronize()
            if k >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        return ts

    rows = []
    with ClockSampler(0) as clk:
        for ctas, fl in ((4, 8), (8, 4)):
            for mib in (16, 32, 64, 128, 256):
                ts = timed(lambda: lib.read_probe(ctypes.c_void_p(buf.data_ptr()), mib << 20,
                                                  ctypes.c_void_p(out.data_ptr()), ctas, fl, st), args.steps)
                m = statistics.mean(ts)
                rows.append({"kernel": f"plain read, {ctas} CTAs x 256 threads per SM, {fl} x 16 B in flight",
                             "mib": mib, "mean_us": round(m, 2), "median_us": round(statistics.median(ts), 2),
                             "gbs": round((mib << 20) / m / 1e3, 1)})
        w = wl.WORKLOADS[wl.HEADLINE]
        x_cpu, mask = wl.make_input(w)
        x = x_cpu.to(dev)
        a = torch.empty(1, device=dev)
        g = torch.empty(1, device=dev)
        ws = torch.zeros(nvfp4.nvfp4_workspace_bytes(), dtype=torch.uint8, device=dev)
        o = nvfp4.make_output(amax=a, global_scale=g)
        for rht in (False, True):
            ts = timed(lambda: nvfp4.nvfp4_amax(x, nvfp4.ROWWISE, rht, mask, o, ws), args.steps)
            m = statistics.mean(ts)
            rows.append({"kernel": f"nvfp4_amax standalone ({'RHT' if rht else 'no RHT'}), {w.name}", "mib": 64,
                         "mean_us": round(m, 2), "median_us": round(statistics.median(ts), 2),
                         "gbs": round((64 << 20) / m / 1e3, 1)})
    return {"read_sweep": rows, "reps": args.steps, "clocks": clk.summary(),
            "l2": "flushed before every call: 512 MiB write + 256 MiB read"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.HEADLINE, choices=list(wl.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget (0 = skip)")
    ap.add_argument("--shape", default=None, help="ROWSxCOLS override of the workload's shape (profiling cases)")
    ap.add_argument("--read-sweep", action="store_true",
                    help="print the plain-read bound after the L2 flush (16..256 MiB) instead of the bench line")
    args = ap.parse_args()
    if args.read_sweep:
        print(json.dumps(read_sweep(args)), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        if args.cpu_seconds > 0 and world == 1:  # the CPU baseline is an N=1 figure
            w = workload_of(args)
            x_cpu, mask = wl.make_input(w)
            res["cpu_baseline"] = cpu_baseline(w, x_cpu, mask, args.cpu_seconds)
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
