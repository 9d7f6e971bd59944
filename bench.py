"""Benchmark of the block-scaled GEMM hot path on GB300.

One step = the whole hot path on one NVFP4 problem: the scale-layout prep of
both operands' row-major scales (one launch), then the persistent
block-scaled GEMM (nvfp4_swizzle_scales2 + nvfp4_gemm_swizzled, the same work
as one nvfp4_gemm call). Default workload: M = N = K = 16384 (the pages' square
sweep shape), inputs resident in HBM, larger than L2.

Prints ONE JSON line (rank 0). Besides the contract's keys it carries the
dominant kernel's roofline (CUDA-event duration of the GEMM launches inside
the timed region), the CPU oracle timed on a bounded sample, the clocks seen
during the timed region, the sustained rate (CUDA-graph replays, median of
15 x 20 iterations, clocks sampled alongside), the host link's copy rates
beside the end-to-end figure, and secondary lines for the FP8 8192^3 GEMM, the
skinny-M sweep (HBM GB/s), the scale swizzle, the NVFP4 quantiser, the
fused epilogue variants (bias, gamma, scattered rows), the grouped (MoE)
GEMM, the NVFP4 x dense-BF16 / FP16 GEMM, and the GEMM from tile-packed
operands against the same GEMM from row-major ones. A compact "summary"
object closes the line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

import workloads  # noqa: E402

# nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): FP4 13.5, FP8 4.5
FP4_PER_BF16 = 13.5 / 2.25
FP8_PER_BF16 = 4.5 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per GEMM launch (dram__bytes_read.sum + dram__bytes_write.sum)
# from one ncu capture, keyed by (plan, workload) and stored with the digest
# of the kernel sources it was taken on (kernel_digest()): once any of them
# changes the figure no longer describes the kernel and traffic reads null.
NCU_TRAFFIC_BYTES: dict[tuple[str, str], tuple[str, float]] = {
    # one-pass capture of the third GEMM launch of
    # bench.py --case nvfp4:16384x16384x16384 --steps 1 --warmup 3
    ("nvfp4_tc2_256x256_s5_acc1", "nvfp4_16384"): ("5a13a3e3fea18730", 1026781696 + 519660800),
}
KERNEL_SOURCES = ("gemm_pair.cu", "gemm_common.cuh", "ptx.cuh", "bsg_internal.h")


def kernel_digest() -> str:
    """sha256 (first 16 hex digits) of the pair kernel's sources."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update((ROOT / "block_scaled_precision_persistent_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(plan: str, workload: str) -> float | None:
    rec = NCU_TRAFFIC_BYTES.get((plan, workload))
    return rec[1] if rec is not None and rec[0] == kernel_digest() else None


def peaks() -> tuple[dict, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        return json.loads(p.read_text()), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (torchrun); N independent replicas, no collective on
# the data path -- the barrier and the max-reduce of the timing only
# ---------------------------------------------------------------------------
def Dist(gpus: int):
    """One process per GPU (torchrun's environment), NCCL; the ranks are
    independent replicas and only the timing crosses them."""
    from block_scaled_precision_persistent_gb300.replicas import Ranks
    return Ranks("nccl", expected_world=gpus)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """SM clock, power and clock-event reasons of this rank's GPU, sampled
    every 5 ms from a background thread through NVML (ctypes on the driver's
    libnvidia-ml; read-only queries), or every 10 ms by nvidia-smi where NVML
    cannot be loaded. The GPU is found by UUID (CUDA's ordinal and NVML's
    index differ under CUDA_VISIBLE_DEVICES)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason* bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int, period_s: float = 0.005):
        self.index = index
        self.period = period_s
        self.rows: list[tuple[float, float, int]] = []     # (sm MHz, power W, reason bits)
        self.max_mhz = None
        self.backend = None
        self.proc = None
        self.file = None
        self.thread = None
        self.stop = False

    # -- NVML -----------------------------------------------------------------
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        want = str(torch.cuda.get_device_properties(self.index).uuid).lower().replace("gpu-", "")
        count = ctypes.c_uint(0)
        lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
        handle = None
        for i in range(count.value):
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
                continue
            buf = ctypes.create_string_buffer(96)
            if lib.nvmlDeviceGetUUID(h, buf, 96) == 0 and \
                    buf.value.decode().lower().replace("gpu-", "") == want:
                handle = h
        if handle is None:
            raise OSError("no NVML device with this GPU's UUID")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        return lib, handle, reasons

    def _nvml_loop(self, lib, handle, reasons):
        import ctypes
        mhz, mw, bits = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self.stop:
            ok = lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(mhz)) == 0
            ok = ok and lib.nvmlDeviceGetPowerUsage(handle, ctypes.byref(mw)) == 0
            ok = ok and reasons(handle, ctypes.byref(bits)) == 0
            if ok:
                self.rows.append((float(mhz.value), mw.value / 1000.0, int(bits.value)))
            time.sleep(self.period)

    def __enter__(self):
        import threading
        try:
            lib, handle, reasons = self._nvml_open()
            self.backend = "nvml, 5 ms"
            self.thread = threading.Thread(target=self._nvml_loop, args=(lib, handle, reasons), daemon=True)
            self.thread.start()
            time.sleep(0.05)
            return self
        except (OSError, AttributeError, RuntimeError):
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        smi_index = ids[self.index] if self.index < len(ids) and ids[self.index].isdigit() else self.index
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={smi_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            self.backend = "nvidia-smi, 10 ms"
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            time.sleep(0.02)
            self.stop = True
            self.thread.join(timeout=5)
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._read_smi()
        return False

    def _read_smi(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        names = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                 "hw_thermal_slowdown": 0x40}
        cols = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in Path(self.file.name).read_text().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9 and num(f[1]) is not None and num(f[3]) is not None:
                bits = sum(names[c] for k, c in enumerate(cols) if f[5 + k] == "Active")
                self.rows.append((num(f[1]), num(f[3]), bits))
                self.max_mhz = num(f[2])
        os.unlink(self.file.name)

    def summary(self) -> dict:
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": ["no samples" if self.backend else "no clock source"]}
        pmax = max(r[1] for r in self.rows)
        loaded = [r for r in self.rows if r[1] > 0.5 * pmax]          # samples under load
        use = loaded or self.rows
        reasons = sorted({name for r in use for bit, name in self.REASONS.items() if r[2] & bit})
        return {"sm_mhz": statistics.median(r[0] for r in use), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min_under_load": min(r[0] for r in use), "reasons": reasons,
                "samples": len(self.rows), "samples_under_load": len(loaded), "power_w_max": round(pmax, 1),
                "power_note": "the driver's averaged board power (about a 1 s window): a burst shorter than "
                              "that reads low; the clock samples are instantaneous",
                "source": self.backend}


# ---------------------------------------------------------------------------
# the hot path
# ---------------------------------------------------------------------------
class Nvfp4Step:
    """Swizzle both scale sets, then the persistent GEMM; GEMM launches are
    bracketed by CUDA events on the launching stream."""

    def __init__(self, w: workloads.Workload, dev):
        import block_scaled_precision_persistent_gb300 as bsg
        self.bsg = bsg
        self.w = w
        p = workloads.make_nvfp4(w, dev)
        self.alpha = p["alpha"]
        self.A, self.sfA, self.B, self.sfB = p["A"], p["sfA"], p["B"], p["sfB"]
        M, N, K = w.M, w.N, w.K
        self.swA = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        self.swB = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        self.D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.launches = 0

    def __call__(self, ev=None):
        b, w = self.bsg, self.w
        st = torch.cuda.current_stream()         # the launching stream (a capture stream in a graph)
        b.nvfp4_swizzle_scales2(w.M, w.N, w.K, self.sfA, self.swA, self.sfB, self.swB, st)
        if ev is not None:
            ev[0].record(st)
        b.nvfp4_gemm_swizzled(w.M, w.N, w.K, self.A, self.swA, self.B, self.swB, self.alpha, self.D, st)
        if ev is not None:
            ev[1].record(st)
        self.launches += 2

    def gemm(self):
        w = self.w
        self.bsg.nvfp4_gemm_swizzled(w.M, w.N, w.K, self.A, self.swA, self.B, self.swB, self.alpha, self.D)

    def plan(self) -> str:
        return self.bsg.bsg_select_plan(0, self.w.M, self.w.N, self.w.K,
                                        torch.cuda.get_device_properties(0).multi_processor_count)


def time_steps(step, steps: int, warmup: int, dist: Dist, gemm_events=True):
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)] if gemm_events else [None] * steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step.launches = 0
    start.record()
    for i in range(steps):
        step(evs[i])
    end.record()
    torch.cuda.synchronize()
    dist.barrier()
    total_ms = start.elapsed_time(end)
    gemm_ms = [a.elapsed_time(b) for a, b in evs] if gemm_events else []
    return total_ms, gemm_ms


def sustained(step: Nvfp4Step, pk: dict, psrc: str, index: int, repeats: int = 15, iters: int = 20) -> dict:
    """The timing practice of the pages (TokenSpeed MLA 2 page, benchmark
    setup): CUDA-graph replays, the median of `repeats` replays of a graph of
    `iters` back-to-back iterations -- here of the whole step (swizzle +
    GEMM) and of the GEMM alone, the two graphs interleaved, with the clocks
    sampled over all of it. Back to back, the GPU runs under its power cap:
    this is the sustained rate, the timed loop's `value` the burst rate."""
    w = step.w
    with ClockSampler(index) as clk:
        us = graph_us({"step": step, "gemm": step.gemm}, iters, repeats)
    clocks = clk.summary()
    if step.bsg.bsg_get_device_status() != step.bsg.BSG_OK:
        raise SystemExit("device status reported an error in the sustained timing")
    peak = pk["bf16_tflops"] * FP4_PER_BF16
    out = {"timing": f"median of {repeats} replays of a CUDA graph of {iters} back-to-back iterations, "
                     "step and GEMM graphs interleaved", "clocks": clocks}
    for k in ("step", "gemm"):
        tf = w.flops / (us[k] * 1e-6) / 1e12
        out[k] = {"us": round(us[k], 2), "tflops": round(tf, 1), "frac_of_9pf": round(tf / 9000.0, 4),
                  "frac": round(tf / peak, 4)}
    out["peak_source"] = f"{psrc} bf16 burst x {FP4_PER_BF16:g}"
    return out


def copy_bandwidth(host: dict, dev_bufs: dict, hD, dD, reps: int = 3) -> dict:
    """Plain pinned-memory copy rates of this host link, for the e2e bound:
    the step's H2D copies alone, its D2H copy alone, and both at once on two
    streams (GB/s, best of `reps`)."""
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    nin = sum(t.numel() * t.element_size() for t in host.values())
    nout = hD.numel() * hD.element_size()

    def timed(which):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if which in ("in", "both"):
                with torch.cuda.stream(h2d):
                    for k, t in host.items():
                        dev_bufs[k].copy_(t, non_blocking=True)
            if which in ("out", "both"):
                with torch.cuda.stream(d2h):
                    hD.copy_(dD, non_blocking=True)
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best
    t_in, t_out, t_both = timed("in"), timed("out"), timed("both")
    return {"h2d_gbs": round(nin / t_in / 1e9, 1), "d2h_gbs": round(nout / t_out / 1e9, 1),
            "both_gbs": round((nin + nout) / t_both / 1e9, 1),
            "copy_bound_ms": round(max(t_in, t_out, t_both) * 1e3, 3)}


def e2e_nvfp4(w: workloads.Workload, step: Nvfp4Step, steps: int, warmup: int) -> dict:
    """The public 10-argument call (nvfp4_gemm: row-major scales, swizzled by
    the library) fed from pinned HOST buffers, as a stream of GEMMs would be:
    two device buffer sets, step i's H2D copies (A, B, both scale sets) on
    one stream while step i-1 computes on a second and step i-2's D returns
    to host memory on a third. Every step's H2D and D2H bytes are inside the
    timed region, which ends when the last D has landed in host memory; the
    returned D is checked bit for bit against the device-only result."""
    bsg = step.bsg
    M, N, K = w.M, w.N, w.K
    host = {k: getattr(step, k).cpu().pin_memory() for k in ("A", "B", "sfA", "sfB")}
    hD = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    slots = [{k: getattr(step, k) for k in ("A", "B", "sfA", "sfB", "D")},
             {k: torch.empty_like(getattr(step, k)) for k in ("A", "B", "sfA", "sfB", "D")}]
    dev = step.D.device
    bsg.bsg_reserve_workspace(dev.index or 0, 2 * (bsg.nvfp4_swizzled_scale_bytes(M, K) + 256))
    h2d, comp, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def issue(i):
        k = i % 2
        t = slots[k]
        h2d.wait_event(comp_done[k])               # the slot's inputs are no longer read
        with torch.cuda.stream(h2d):
            for name in ("A", "B", "sfA", "sfB"):
                t[name].copy_(host[name], non_blocking=True)
        in_ready[k].record(h2d)
        comp.wait_event(in_ready[k])
        comp.wait_event(out_done[k])               # the slot's D has been copied out
        bsg.nvfp4_gemm(M, N, K, t["A"], t["sfA"], t["B"], t["sfB"], step.alpha, t["D"], comp)
        comp_done[k].record(comp)
        d2h.wait_event(comp_done[k])
        with torch.cuda.stream(d2h):
            hD[k].copy_(t["D"], non_blocking=True)
        out_done[k].record(d2h)

    for i in range(warmup):
        issue(i)
    torch.cuda.synchronize()
    # five timed runs of `steps` steps each, the median per step: the host
    # link and host memory are shared with the rest of the machine, and a
    # run can catch another job's copies
    runs = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(h2d)
        for i in range(steps):
            issue(i)
        d2h.wait_event(comp_done[(steps - 1) % 2])
        b.record(d2h)
        torch.cuda.synchronize()
        runs.append(a.elapsed_time(b) / steps)
    ms = statistics.median(runs)
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error in the e2e run")
    ref = step.D.view(torch.int16).cpu()
    for k in range(min(2, steps)):
        if not torch.equal(hD[k].view(torch.int16), ref):
            raise SystemExit("e2e: D copied back differs from the device-only result")
    h2d_bytes = sum(t.numel() * t.element_size() for t in host.values())
    d2h_bytes = hD[0].numel() * hD[0].element_size()
    link = copy_bandwidth(host, slots[1], hD[1], slots[1]["D"])
    del slots[1]
    # the pipeline overlaps the GEMM with both copies, so a step cannot take
    # less than its copies alone (both directions at once): the bound
    link["frac_of_copy_bound"] = round(link["copy_bound_ms"] / ms, 4)
    return {"value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "pipelined": "two buffer sets; H2D, compute and D2H on three streams",
            "runs_ms_per_step": [round(r, 4) for r in runs], "timing": "median of five timed runs", "host_link": link}


def secondary_fp8(dev, steps: int, warmup: int, pk: dict, psrc: str) -> dict:
    import block_scaled_precision_persistent_gb300 as bsg
    w = workloads.WORKLOADS["fp8_8192"]
    q = workloads.make_fp8(w, dev)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        bsg.fp8_gemm(w.M, w.N, w.K, q["A"], None, q["B"], None, q["alpha"], D, s)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        a.record(s)
        bsg.fp8_gemm(w.M, w.N, w.K, q["A"], None, q["B"], None, q["alpha"], D, s)
        b.record(s)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    tf = w.flops / (ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"] * FP8_PER_BF16
    return {"workload": w.name, "plan": bsg.bsg_select_plan(1, w.M, w.N, w.K, 152),
            "ms": ms, "tflops": tf, "roofline_peak_tflops": peak, "frac": tf / peak,
            "peak_source": f"{psrc} bf16 burst x {FP8_PER_BF16:g} (nominal FP8/BF16)"}


def secondary_skinny(dev, steps: int, pk: dict, psrc: str) -> dict:
    """Each cell timed cold and back to back: a CUDA graph of one launch per
    buffer set, the sets rotated over > 4x L2 so every launch reads its
    weights from HBM, replayed `steps` times; per-launch time = median replay
    time / launches in the graph."""
    import block_scaled_precision_persistent_gb300 as bsg
    out = {}
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for name, w in workloads.WORKLOADS.items():
        if "skinny" not in name:
            continue
        p = workloads.make_nvfp4(w, dev)
        M, N, K = w.M, w.N, w.K
        swA = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        swB = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, p["sfA"], swA)
        bsg.nvfp4_swizzle_scales(N, K, p["sfB"], swB)
        per = w.algorithmic_bytes
        copies = max(2, int(4 * l2 // per) + 1)
        sets = [(p["A"].clone(), swA.clone(), p["B"].clone(), swB.clone(),
                 torch.empty((M, N), dtype=torch.bfloat16, device=dev)) for _ in range(copies)]
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            for A, sa, B, sb, D in sets[:3]:
                bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, p["alpha"], D)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for A, sa, B, sb, D in sets:
                bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, p["alpha"], D)
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / copies)
        if bsg.bsg_get_device_status() != bsg.BSG_OK:
            raise RuntimeError(f"device status set during skinny cell {name}")
        us = statistics.median(ts) * 1e3
        # warm L2: the same graph shape over one buffer set, so weights stay in L2
        gw = torch.cuda.CUDAGraph()
        A, sa, B, sb, D = sets[0]
        with torch.cuda.graph(gw):
            for _ in range(copies):
                bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, p["alpha"], D)
        gw.replay()
        torch.cuda.synchronize()
        tw = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gw.replay()
            b.record()
            torch.cuda.synchronize()
            tw.append(a.elapsed_time(b) / copies)
        us_warm = statistics.median(tw) * 1e3
        # the same cold graph with programmatic dependent launch: each
        # launch's prologue overlaps the previous launch's tail (mode 1);
        # mode 2 also starts reading the weights' codes before the wait
        # (no launch here writes another's weights)
        us_pdl_mode = {}
        for mode in (1, 2):
            bsg.bsg_set_pdl(mode)
            try:
                gp = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gp):
                    for A, sa, B, sb, D in sets:
                        bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, p["alpha"], D)
            finally:
                bsg.bsg_set_pdl(False)
            gp.replay()
            torch.cuda.synchronize()
            tp = []
            for _ in range(steps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                gp.replay()
                b.record()
                torch.cuda.synchronize()
                tp.append(a.elapsed_time(b) / copies)
            if bsg.bsg_get_device_status() != bsg.BSG_OK:
                raise RuntimeError(f"device status set during the PDL run of skinny cell {name}")
            us_pdl_mode[mode] = statistics.median(tp) * 1e3
            del gp
        us_pdl, us_pdl_w = us_pdl_mode[1], us_pdl_mode[2]
        gbs = per / (us * 1e-6) / 1e9
        ideal_us = max(per / (pk["hbm_gbs"] * 1e9), w.flops / (pk["bf16_tflops"] * FP4_PER_BF16 * 1e12)) * 1e6
        out[f"m{M}_n{N}_k{K}"] = {"plan": bsg.bsg_select_plan(0, M, N, K, sms), "us": round(us, 3),
                                  "hbm_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                                  "ideal_us": round(ideal_us, 3), "frac_roofline": round(ideal_us / us, 4),
                                  "us_warm_l2": round(us_warm, 3), "us_pdl": round(us_pdl, 3),
                                  "hbm_gbs_pdl": round(per / (us_pdl * 1e-6) / 1e9, 1),
                                  "us_pdl_weights_early": round(us_pdl_w, 3),
                                  "frac_hbm_pdl_weights_early": round(per / (us_pdl_w * 1e-6) / 1e9 / pk["hbm_gbs"], 4)}
        del g, gw, sets
    return {"cells": out, "peak_hbm_gbs": pk["hbm_gbs"], "peak_source": psrc,
            "timing": "cold L2 (buffer sets rotated over > 4x L2), CUDA graph of back-to-back launches, "
                      "median over replays of graph time / launches; us_warm_l2: the same over one "
                      "buffer set (weights L2-resident); us_pdl: the cold graph with programmatic "
                      "dependent launch; us_pdl_weights_early: the same with bsg_set_pdl(2), the weights' "
                      "codes read before each launch waits for the previous one"}


def secondary_quantize(dev, steps: int, pk: dict, psrc: str) -> dict:
    """Two-level NVFP4 quantisation of a BF16 [16384][16384] matrix (one
    operand of the headline GEMM): memset + amax pass + quantise pass.
    Algorithmic bytes: X read twice (the global amax precedes every block's
    scale), codes and swizzled scales written. X (512 MiB) exceeds L2."""
    import block_scaled_precision_persistent_gb300 as bsg
    rows, K = 16384, 16384
    x = torch.randn((rows, K), device=dev, dtype=torch.float32).to(torch.bfloat16)
    packed = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    swz = torch.empty(bsg.nvfp4_swizzled_scale_bytes(rows, K), dtype=torch.uint8, device=dev)
    gl = torch.empty(2, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream()
    for _ in range(3):
        bsg.nvfp4_quantize(rows, K, x, packed, swz, None, gl, s)
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        bsg.nvfp4_quantize(rows, K, x, packed, swz, None, gl, s)
        b.record(s)
        evs.append((a, b))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    # the same with the codes written in the tile-packed layout
    evs = []
    for i in range(steps + 3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        bsg.nvfp4_quantize_tiles(rows, K, x, packed, swz, None, gl, s)
        b.record(s)
        if i >= 3:
            evs.append((a, b))
    torch.cuda.synchronize()
    us_tiles = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    moved = 2 * (2 * rows * K) + rows * K // 2 + bsg.nvfp4_swizzled_scale_bytes(rows, K)
    gbs = moved / (us * 1e-6) / 1e9
    return {"shape": f"bf16 {rows} x {K}", "us": round(us, 2), "gb_s": round(gbs, 1),
            "frac_hbm": round(gbs / pk["hbm_gbs"], 4), "algorithmic_bytes": moved, "peak_source": psrc,
            "us_tile_packed_codes": round(us_tiles, 2),
            "launches": 2, "timing": "median per-call CUDA events (memset + 2 kernels), X > L2"}


def graph_us(calls: dict, launches: int, replays: int) -> dict:
    """Per-launch device time of each call in `calls` (name -> callable): one
    CUDA graph of `launches` back-to-back calls per name (captured after
    three warm calls on a side stream), the graphs then replayed in turn,
    round after round, so that clock or power drift falls on every variant
    alike; median over `replays` rounds of replay time / launches. Keeps the
    host's per-call cost (tensor-map encoding, launch) out of the number."""
    side = torch.cuda.Stream()
    graphs = {}
    for name, call in calls.items():
        with torch.cuda.stream(side):
            for _ in range(3):
                call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(launches):
                call()
        g.replay()
        torch.cuda.synchronize()
        graphs[name] = g
    ts = {name: [] for name in calls}
    for _ in range(replays):
        for name, g in graphs.items():
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            g.replay()
            t1.record()
            torch.cuda.synchronize()
            ts[name].append(t0.elapsed_time(t1) * 1e3 / launches)
    del graphs
    return {name: statistics.median(v) for name, v in ts.items()}


def secondary_epilogue(dev, step: Nvfp4Step, steps: int, pk: dict, psrc: str) -> dict:
    """The NVFP4 GEMM with the fused epilogue variants (nvfp4_gemm_ex): the
    plain call, bias + gamma, and bias + gamma + a scatter permutation of
    the rows, on the same resident operands: 16384^3 (the headline step's
    buffers, larger than L2), 4096^3, and the 64 x 3072 x 3072 skinny cell
    (weights L2-resident). Timed as CUDA graphs of back-to-back launches
    (graph_us); vs_plain = plain time / variant time."""
    import block_scaled_precision_persistent_gb300 as bsg
    step()                                     # swizzled scales of the step are current
    torch.cuda.synchronize()
    keep = []

    def problem(name):
        w = workloads.WORKLOADS[name]
        p = workloads.make_nvfp4(w, dev)
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(w.M, w.K), dtype=torch.uint8, device=dev)
        sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(w.N, w.K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(w.M, w.K, p["sfA"], sa)
        bsg.nvfp4_swizzle_scales(w.N, w.K, p["sfB"], sb)
        D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        keep.append((p, sa, sb, D))
        return (w.M, w.N, w.K, p["A"], sa, p["B"], sb, p["alpha"], D, w.std)

    shapes = {
        "nvfp4_16384": ((step.w.M, step.w.N, step.w.K, step.A, step.swA, step.B, step.swB, step.alpha,
                         step.D, step.w.std), 4),
        "nvfp4_4096": (problem("nvfp4_4096"), 32),
        "nvfp4_skinny_m64_n3072_k3072": (problem("nvfp4_skinny_m64_n3072_k3072"), 32),
    }
    out = {}
    for wname, ((M, N, K, A, sa, B, sb, alpha, D, std), launches) in shapes.items():
        # let the clock recover from the previous shape's power-capped
        # graphs, so that each shape runs at its own clock
        torch.cuda.synchronize()
        time.sleep(0.5)
        e = workloads.make_epilogue(M, N, seed=3, bias_std=float(K) ** 0.5 * std * std, device=dev)
        variants = {"plain": (None, None, None), "bias": (e["bias"], None, None), "gamma": (None, e["gamma"], None),
                    "bias_gamma": (e["bias"], e["gamma"], None),
                    "bias_gamma_scatter": (e["bias"], e["gamma"], e["scatter"])}
        calls = {v: (lambda b=b, g=g, sc=sc: bsg.nvfp4_gemm_ex(M, N, K, A, sa, B, sb, alpha, b, g, sc, M, D))
                 for v, (b, g, sc) in variants.items()}

        def plain_pdl():
            # the plain call with programmatic dependent launch: each launch's
            # prologue overlaps the previous one's tail (reported beside the
            # plain figure, which keeps it off)
            bsg.bsg_set_pdl(True)
            try:
                bsg.nvfp4_gemm_ex(M, N, K, A, sa, B, sb, alpha, None, None, None, M, D)
            finally:
                bsg.bsg_set_pdl(False)
        calls["plain_pdl"] = plain_pdl
        times = graph_us(calls, launches, steps)
        cells = {v: {"us": round(us, 3), "tflops": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1)}
                 for v, us in times.items()}
        for v in cells.values():
            v["vs_plain"] = round(cells["plain"]["us"] / v["us"], 4)
        out[wname] = dict(cells, plan=bsg.bsg_select_plan(0, M, N, K, 152), launches_per_graph=launches)
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error in the epilogue-variant timing")
    del keep
    peak = pk["bf16_tflops"] * FP4_PER_BF16
    return {"shapes": out, "roofline_peak_tflops": peak, "peak_source": psrc,
            "timing": "CUDA graph of back-to-back launches per variant, the variants' graphs replayed in "
                      "turn, median over rounds of graph time / launches; "
                      "operands resident (16384^3 larger than L2; 4096^3 and the skinny cell L2-resident)"}


class GroupedProblem:
    """The MoE workload on the device: routing offsets, the per-slice
    swizzled A scales, the experts' swizzled B scales, D in token order."""

    def __init__(self, w, dev):
        import block_scaled_precision_persistent_gb300 as bsg
        self.bsg, self.w = bsg, w
        offs, dst = workloads.routing(w.E, w.tokens, w.top_k, seed=1)
        self.offs, self.dst = offs.to(dev), dst.to(dev)
        p = workloads.make_grouped(w.E, w.M, w.N, w.K, seed=1, device=dev)
        self.A, self.B, self.alpha = p["A"], p["B"], p["alpha"]
        self.sa = torch.empty(bsg.nvfp4_grouped_scale_bytes(w.E, w.M, w.K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales_grouped(w.E, w.M, w.K, self.offs, p["sfA"], self.sa)
        # the experts' [E*N][K/16] scales swizzle as one matrix (N % 128 == 0)
        assert w.N % 128 == 0
        self.sb = torch.empty(w.E * bsg.nvfp4_swizzled_scale_bytes(w.N, w.K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(w.E * w.N, w.K, p["sfB"].reshape(w.E * w.N, -1), self.sb)
        self.D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        del p

    def __call__(self, scatter=True):
        w = self.w
        self.bsg.nvfp4_grouped_gemm(w.E, w.M, w.N, w.K, self.A, self.sa, self.B, self.sb, self.offs, self.alpha,
                                    None, None, self.dst if scatter else None, w.M, self.D)


def secondary_grouped(dev, steps: int, pk: dict, psrc: str) -> dict:
    """The grouped (MoE) NVFP4 GEMM: 64 experts, 1024 tokens x top-8 (8192
    routed rows, ~128 per expert), 4096 x 7168 weights per expert, D written
    in token order (scatter) and in expert order. HBM-bound: algorithmic
    bytes = packed A + all experts' packed weights and scales + BF16 D
    (1.16 GB, of which the weights 1.09 GB), larger than L2. Timed as
    interleaved CUDA graphs of back-to-back launches (graph_us)."""
    import block_scaled_precision_persistent_gb300 as bsg
    w = workloads.GROUPED_WORKLOADS["moe_e64_t1024_k8"]
    g = GroupedProblem(w, dev)
    times = graph_us({"scatter": lambda: g(True), "expert_order": lambda: g(False)}, 8, steps)
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error in the grouped GEMM timing")
    out = {}
    for k, us in times.items():
        gbs = w.algorithmic_bytes / (us * 1e-6) / 1e9
        out[k] = {"us": round(us, 2), "tflops": round(w.flops / (us * 1e-6) / 1e12, 1), "hbm_gbs": round(gbs, 1),
                  "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
    ideal = max(w.algorithmic_bytes / (pk["hbm_gbs"] * 1e9), w.flops / (pk["bf16_tflops"] * FP4_PER_BF16 * 1e12))
    g()
    plan = bsg.bsg_last_plan_name()
    del g
    # the pages' own ragged matrix multiplies routed NVFP4 rows by dense
    # 16-bit expert weights: the same routing with BF16 weights [E][N][K]
    # (nvfp4_dense_grouped_gemm), D in token order
    offs, dst = workloads.routing(w.E, w.tokens, w.top_k, seed=1)
    offs, dst = offs.to(dev), dst.to(dev)
    pd = workloads.make_dense_grouped(w.E, w.M, w.N, w.K, seed=1, device=dev)
    sa = torch.empty(bsg.nvfp4_grouped_scale_bytes(w.E, w.M, w.K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales_grouped(w.E, w.M, w.K, offs, pd["sfA"], sa)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)

    def dense_call():
        bsg.nvfp4_dense_grouped_gemm(w.E, w.M, w.N, w.K, pd["A"], sa, pd["B"], offs, pd["alpha"], None, None, dst,
                                     w.M, D)
    us = graph_us({"dense": dense_call}, 4, steps)["dense"]
    dense_call()
    dplan = bsg.bsg_last_plan_name()
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error in the grouped dense GEMM timing")
    dbytes = w.M * w.K * 9 // 16 + w.E * w.N * w.K * 2 + w.M * w.N * 2
    dgbs = dbytes / (us * 1e-6) / 1e9
    dense = {"plan": dplan, "us": round(us, 2), "tflops": round(w.flops / (us * 1e-6) / 1e12, 1),
             "hbm_gbs": round(dgbs, 1), "frac_hbm": round(dgbs / pk["hbm_gbs"], 4), "algorithmic_bytes": dbytes,
             "ideal_us": round(max(dbytes / (pk["hbm_gbs"] * 1e9), w.flops / (pk["bf16_tflops"] * 1e12)) * 1e6, 2)}
    del pd, sa, D
    return {"workload": w.name, "E": w.E, "M": w.M, "N": w.N, "K": w.K, "plan": plan, "variants": out,
            "ideal_us": round(ideal * 1e6, 2), "algorithmic_bytes": w.algorithmic_bytes, "peak_hbm_gbs": pk["hbm_gbs"],
            "peak_source": psrc, "dense_bf16_weights": dense,
            "timing": "CUDA graph of 8 back-to-back launches per variant, replayed in turn; median per launch"}


def secondary_dense(dev, steps: int, pk: dict, psrc: str) -> dict:
    """NVFP4 activations x dense weights (nvfp4_dense_gemm with BF16 B,
    nvfp4_dense_f16_gemm with FP16 B): 8192^3 in both, an 8192 x 256 x 8192
    weight GEMM (the pages' case has N = 256) in BF16, and the K-ragged form
    (nvfp4_dense_kgrouped_gemm) over eight slices of K. A is expanded to
    B's type on the fly and the 16-bit tensor core computes, so the roofline
    is the measured BF16 GEMM peak (FP16 runs at the same nominal rate).
    CUDA graphs, median per launch."""
    import block_scaled_precision_persistent_gb300 as bsg
    out = {}
    for (M, N, K), launches, f16 in (((8192, 8192, 8192), 4, False), ((8192, 8192, 8192), 4, True),
                                     ((8192, 256, 8192), 16, False)):
        p = workloads.make_dense(M, N, K, seed=1, device=dev, b_dtype=torch.float16 if f16 else torch.bfloat16)
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, p["sfA"], sa)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        dense = bsg.nvfp4_dense_f16_gemm if f16 else bsg.nvfp4_dense_gemm

        def call():
            dense(M, N, K, p["A"], sa, p["B"], p["alpha"], None, None, None, M, D)
        us = graph_us({"dense": call}, launches, steps)["dense"]
        call()
        plan = bsg.bsg_last_plan_name()
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        out[f"{M}x{N}x{K}" + ("_f16" if f16 else "")] = {"plan": plan, "us": round(us, 2), "tflops": round(tf, 1),
                                                         "frac_bf16": round(tf / pk["bf16_tflops"], 4)}
        del p, sa, D
    # K-ragged (inner-expert): K = 8192 split into 8 uneven slices (whole
    # 64-element blocks, seeded), each slice its own 4096 x 4096 output
    M = N = 4096
    K = 8192
    import numpy as np
    rng = np.random.default_rng(8)
    cuts = np.sort(rng.choice(np.arange(1, K // 64), 7, replace=False)) * 64
    koffs = torch.tensor([0, *cuts.tolist(), K], dtype=torch.int32, device=dev)
    p = workloads.make_dense(M, N, K, seed=2, device=dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"], sa)
    D = torch.empty((8, M, N), dtype=torch.bfloat16, device=dev)

    def kcall():
        bsg.nvfp4_dense_kgrouped_gemm(8, M, N, K, p["A"], sa, p["B"], koffs, p["alpha"], None, None, D)
    us = graph_us({"kragged": kcall}, 4, steps)["kragged"]
    kcall()
    kplan = bsg.bsg_last_plan_name()
    flops = 2.0 * M * N * K
    kbytes = M * K * 9 // 16 + N * K * 2 + 8 * M * N * 2
    out["kragged_e8_4096x4096x8192"] = {
        "plan": kplan, "us": round(us, 2), "tflops": round(flops / (us * 1e-6) / 1e12, 1),
        "frac_bf16": round(flops / (us * 1e-6) / 1e12 / pk["bf16_tflops"], 4),
        "hbm_gbs": round(kbytes / (us * 1e-6) / 1e9, 1), "slices_k": [0, *cuts.tolist(), K],
        "note": "eight outputs of 4096 x 4096 (268 MB of D); FLOPs are those of the whole K"}
    del p, sa, D
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error in the dense GEMM timing")
    return {"shapes": out, "roofline_peak_tflops": pk["bf16_tflops"],
            "peak_source": f"{psrc} bf16 burst (the MMA is kind::f16 on BF16 operands)",
            "timing": "CUDA graph of back-to-back launches, median over replays per launch"}


def secondary_packed(dev, step: Nvfp4Step, pk: dict, psrc: str) -> dict:
    """The headline shape with A and B in the tile-packed layout
    (nvfp4_gemm_packed: operand tiles by contiguous bulk copies) against the
    same GEMM from row-major operands (tensor-map boxes), as interleaved
    CUDA graphs; plus the cost of packing one operand (A, as activations
    would be each step; weights are packed once)."""
    import block_scaled_precision_persistent_gb300 as bsg
    w = step.w
    M, N, K = w.M, w.N, w.K
    s = torch.cuda.current_stream()
    step()                                     # swizzled scales in step.swA / step.swB
    ap = torch.empty(bsg.nvfp4_packed_operand_bytes(M, K), dtype=torch.uint8, device=dev)
    bp = torch.empty(bsg.nvfp4_packed_operand_bytes(N, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_pack_operand(M, K, step.A, ap, s)
    bsg.nvfp4_pack_operand(N, K, step.B, bp, s)
    torch.cuda.synchronize()
    calls = {
        "tensor_map": lambda: bsg.nvfp4_gemm_swizzled(M, N, K, step.A, step.swA, step.B, step.swB, step.alpha,
                                                      step.D),
        "packed": lambda: bsg.nvfp4_gemm_packed(M, N, K, ap, step.swA, bp, step.swB, step.alpha, step.D),
        "pack_a": lambda: bsg.nvfp4_pack_operand(M, K, step.A, ap),
    }
    us = graph_us(calls, 8, 5)
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error in the packed-operand timing")
    tf = {k: w.flops / (us[k] * 1e-6) / 1e12 for k in ("tensor_map", "packed")}
    pack_bytes = 2 * (M * K // 2)
    gbs = pack_bytes / (us["pack_a"] * 1e-6) / 1e9
    del ap, bp
    return {"shape": f"{M}x{N}x{K}", "plan": "nvfp4_tc2_256x256_s5_acc1_packed",
            "us": {k: round(v, 2) for k, v in us.items()},
            "tflops_tensor_map": round(tf["tensor_map"], 1), "tflops_packed": round(tf["packed"], 1),
            "packed_over_tensor_map": round(us["tensor_map"] / us["packed"], 4),
            "tflops_packed_incl_pack_a": round(w.flops / ((us["packed"] + us["pack_a"]) * 1e-6) / 1e12, 1),
            "pack_a_gb_s": round(gbs, 1), "pack_a_frac_hbm": round(gbs / pk["hbm_gbs"], 4), "peak_source": psrc,
            "timing": "interleaved CUDA graphs of 8 back-to-back launches, median of 5 rounds"}


def secondary_swizzle(dev, steps: int, pk: dict, psrc: str) -> dict:
    """The scale-layout prep alone (timed separately from the GEMM): one
    operand's row-major [16384][1024] E4M3 scales into the swizzled layout;
    bytes = read + write. Inputs rotate over > 4x L2 (cold)."""
    import block_scaled_precision_persistent_gb300 as bsg
    rows, K = 16384, 16384
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    nbytes = rows * (K // 16)
    copies = max(2, int(4 * l2 // (2 * nbytes)) + 1)
    src = [torch.randint(0, 256, (rows, K // 16), dtype=torch.uint8, device=dev) for _ in range(copies)]
    dst = [torch.empty(bsg.nvfp4_swizzled_scale_bytes(rows, K), dtype=torch.uint8, device=dev)
           for _ in range(copies)]
    s = torch.cuda.current_stream()
    for i in range(3):
        bsg.nvfp4_swizzle_scales(rows, K, src[i % copies], dst[i % copies], s)
    torch.cuda.synchronize()
    # per-launch events around single calls: the host's per-call time can
    # exceed the kernel's, so these include the gaps it leaves
    evs = []
    for i in range(max(steps, copies)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        bsg.nvfp4_swizzle_scales(rows, K, src[i % copies], dst[i % copies], s)
        b.record(s)
        evs.append((a, b))
    torch.cuda.synchronize()
    us_events = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    # the kernel's own time: a CUDA graph of back-to-back launches over the
    # rotated buffers, median over replays, per launch
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        bsg.nvfp4_swizzle_scales(rows, K, src[0], dst[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(copies):
            bsg.nvfp4_swizzle_scales(rows, K, src[i], dst[i])
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(5, steps)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / copies)
    del g
    us = statistics.median(ts)
    moved = nbytes + bsg.nvfp4_swizzled_scale_bytes(rows, K)
    gbs = moved / (us * 1e-6) / 1e9
    return {"shape": f"{rows} rows x K={K}", "us": round(us, 3), "gb_s": round(gbs, 1),
            "frac_hbm": round(gbs / pk["hbm_gbs"], 4), "peak_source": psrc, "us_per_call_events": round(us_events, 3),
            "timing": "cold (inputs rotated over > 4x L2): a CUDA graph of back-to-back launches, median per launch; "
                      "us_per_call_events: per-call CUDA events around single calls"}


def cpu_baseline(w: workloads.Workload, p_host: dict, budget_s: float = 15.0) -> dict:
    """The oracle, as it stands, on a bounded sample of the same workload:
    a number of complete output rows (all N columns, full K)."""
    import oracle
    o = oracle.get()
    threads = oracle.default_threads()
    args = (p_host["A"], p_host["sfA"], p_host["B"], p_host["sfB"], p_host["alpha"], w.K)
    # calibrate on one row per thread, then size the sample to ~budget_s
    t = time.perf_counter()
    o.nvfp4_gemm(*args, rows=list(range(threads)), nthreads=threads)
    per_round = max(time.perf_counter() - t, 1e-3)       # seconds per `threads` rows
    rows = int(budget_s / per_round) * threads
    rows = max(threads, min(w.M, rows))
    sel = list(range(0, w.M, max(1, w.M // rows)))[:rows]
    t = time.perf_counter()
    o.nvfp4_gemm(*args, rows=sel, nthreads=threads)
    dt = time.perf_counter() - t
    flops = 2.0 * len(sel) * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(sel)} of {w.M} output rows x all {w.N} columns, K={w.K} "
                      f"({dt:.1f} s of CPU work)", "seconds": dt, "cpu": host_cpu(),
            "full_matrix_seconds_extrapolated": round(dt * w.M / len(sel), 1)}


def host_cpu() -> dict:
    """The host's CPU as /proc/cpuinfo names it (x86: "model name"; Arm:
    implementer and part codes), its online CPU count and the CPUs this
    process may run on."""
    model = None
    ids = {}
    try:
        for line in Path("/proc/cpuinfo").read_text().splitlines():
            k, _, v = line.partition(":")
            k, v = k.strip(), v.strip()
            if k == "model name" and not model:
                model = v
            elif k in ("CPU implementer", "CPU part") and k not in ids:
                ids[k] = v
    except OSError:
        pass
    if not model and ids:
        model = "implementer {} part {}".format(ids.get("CPU implementer", "?"), ids.get("CPU part", "?"))
    return {"model": model or platform.processor() or platform.machine(), "nproc": os.cpu_count(),
            "affinity": len(os.sched_getaffinity(0))}


def cpu_configs() -> dict:
    """The oracle, as it stands, on the whole of each smaller configuration
    (every output element): NVFP4 256^3 and 4096^3, FP8 8192^3 and the twelve
    skinny cells. Inputs are generated on the host with the same seeded
    recipes as the GPU runs. Opt-in (--cpu-configs): about a minute of CPU."""
    import oracle
    o = oracle.get()
    threads = oracle.default_threads()
    out = {}
    names = ["nvfp4_256", "nvfp4_4096", "fp8_8192"] + [n for n in workloads.WORKLOADS if "skinny" in n]
    for name in names:
        w = workloads.WORKLOADS[name]
        if w.kind == "fp8":
            q = workloads.make_fp8(w, "cpu")
            args = (q["A"].numpy(), q["B"].numpy(), q["alpha"])
            t = time.perf_counter()
            o.fp8_gemm(*args, nthreads=threads)
        else:
            p = workloads.make_nvfp4(w, "cpu")
            args = (p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(), p["sfB"].numpy(), p["alpha"], w.K)
            t = time.perf_counter()
            o.nvfp4_gemm(*args, nthreads=threads)
        dt = time.perf_counter() - t
        out[name] = {"seconds": round(dt, 3), "gflops": round(w.flops / dt / 1e9, 2)}
    return {"cores": threads, "kind": "oracle", "scope": "every output element", "configs": out}


def ingress_roofline(bsg, w: workloads.Workload, plan: str, gemm_ms: float, clocks: dict) -> dict | None:
    """The headline kernel against the rate at which an SM can take operands
    in: bytes each CTA must load per k-block (its 128 A rows and BN/2 B rows
    of 128 bytes, A's 2 KiB and B's BN/128 x 2 KiB of block scales) times the
    k-blocks a CTA runs on average, per SM cycle, against the probe's
    measured ceiling (bsg_measure_ingress, 32 MiB L2-resident source)."""
    if not plan.startswith("nvfp4_tc2_256x"):
        return None
    bn = int(plan.split("_")[2].split("x")[1])
    per_kblock = 128 * 128 + (bn // 2) * 128 + 2048 + (bn // 128) * 2048
    tiles = -(-w.M // 256) * -(-w.N // bn)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    kblocks_per_cta = 2.0 * tiles * (w.K // 256) / grid
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz")
    if not mhz:
        return None
    achieved = kblocks_per_cta * per_kblock / (gemm_ms * 1e-3 * mhz * 1e6)
    peak, total = bsg.bsg_measure_ingress(32 << 20, 4)
    box, _ = bsg.bsg_measure_ingress(32 << 20, 4, tensor_boxes=True)
    return {"bound": "per-SM operand ingress", "bytes_per_kblock_per_cta": per_kblock,
            "achieved_bytes_per_cycle_per_sm": round(achieved, 2), "peak_bytes_per_cycle_per_sm": round(peak, 2),
            "frac": round(achieved / peak, 4), "probe_total_gbs": round(total, 1),
            "tensor_box_bytes_per_cycle_per_sm": round(box, 2), "frac_of_tensor_box": round(achieved / box, 4),
            "peak_note": "peak: contiguous bulk copies; tensor_box: 128-row x 128-byte tensor-map boxes, "
                         "the load the kernel issues for its operand tiles",
            "cycles": f"SM clock {mhz:.0f} MHz (median sampled under load)"}


def host_copy(step: Nvfp4Step) -> dict:
    return {"A": step.A.cpu().numpy(), "sfA": step.sfA.cpu().numpy(), "B": step.B.cpu().numpy(),
            "sfB": step.sfB.cpu().numpy(), "alpha": step.alpha}


def run_ours(args, dist: Dist) -> None:
    import __graft_entry__
    if dist.local == 0:
        __graft_entry__.build()
    dist.barrier()
    import block_scaled_precision_persistent_gb300 as bsg
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    pk, psrc = peaks()
    w = workloads.WORKLOADS[args.workload]
    step = Nvfp4Step(w, dev)
    # one correctness gate before timing: status word clean after a warm call
    step()
    torch.cuda.synchronize()
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error on the warm-up call")

    with ClockSampler(dist.local) as clk:
        total_ms, gemm_ms = time_steps(step, args.steps, args.warmup, dist)
    clocks = clk.summary()
    sus = sustained(step, pk, psrc, dist.local) if dist.rank == 0 else None
    launches = step.launches
    ms = dist.max(total_ms / args.steps)
    value = dist.world * w.flops / (ms * 1e-3) / 1e12
    gemm_avg = statistics.mean(gemm_ms)
    achieved = w.flops / (gemm_avg * 1e-3) / 1e12
    peak = pk["bf16_tflops"] * FP4_PER_BF16
    plan = step.plan()
    traffic = ncu_traffic(plan, w.name)
    ingress = None
    if dist.rank == 0:
        ingress = ingress_roofline(bsg, w, plan, gemm_avg, clocks)

    e2e = None
    if not args.no_e2e:
        e2e = e2e_nvfp4(w, step, max(4, min(args.steps, 10)), 2)
        e2e["ms_per_step"] = dist.max(e2e["ms_per_step"])
        e2e["value"] = dist.world * w.flops / (e2e["ms_per_step"] * 1e-3) / 1e12
    secondary = {}
    if not args.no_secondary:
        secondary["fp8"] = secondary_fp8(dev, max(3, args.steps), args.warmup, pk, psrc)
        secondary["skinny"] = secondary_skinny(dev, 20, pk, psrc)
        secondary["swizzle"] = secondary_swizzle(dev, 20, pk, psrc)
        secondary["quantize"] = secondary_quantize(dev, 20, pk, psrc)
        secondary["epilogue"] = secondary_epilogue(dev, step, 10, pk, psrc)
        secondary["grouped"] = secondary_grouped(dev, 15, pk, psrc)
        secondary["dense"] = secondary_dense(dev, 10, pk, psrc)
        secondary["packed"] = secondary_packed(dev, step, pk, psrc)
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, host_copy(step), args.cpu_seconds)
        cpu["gpu_over_oracle"] = round(value / cpu["value"], 1)
        if args.cpu_configs:
            cpu["full_configs"] = cpu_configs()

    line = {
        "metric": "NVFP4 GEMM TFLOPS at 16384^3 (whole hot path: scale prep + persistent GEMM)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3 block scales) -> f32 acc -> bf16",
        "data": "synthetic (seeded N(0,1) -> two-level NVFP4 quantisation)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "plan": plan,
                   "l2": "inputs larger than L2 (A+B+scales+D = 800 MiB)",
                   "parallelism": f"replicas x{dist.world}"},
        "impl": "ours",
        "gemm_only": {"ms": round(gemm_avg, 4), "tflops": round(achieved, 2)},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": plan,
                     "peak_source": f"{psrc} bf16 burst {pk['bf16_tflops']} x {FP4_PER_BF16:g} "
                                    "(nominal FP4/BF16 dense ratio)",
                     "frac_of_9pf": round(achieved / 9000.0, 4), "ingress": ingress},
        "e2e": None if e2e is None else
               {k: (round(v, 4) if isinstance(v, float) else v) for k, v in e2e.items()},
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "sustained": sus,
        "secondary": secondary,
    }
    # compact figures last on the line, where a record that keeps only the
    # line's end still holds them
    summary = {"gemm_burst_tflops": round(achieved, 1), "gemm_burst_frac_9pf": round(achieved / 9000.0, 4)}
    if sus is not None:
        summary.update(gemm_sustained_us=sus["gemm"]["us"], gemm_sustained_frac_9pf=sus["gemm"]["frac_of_9pf"],
                       step_sustained_us=sus["step"]["us"], sustained_sm_mhz=sus["clocks"].get("sm_mhz"))
    if "fp8" in secondary:
        f = secondary["fp8"]
        summary.update(fp8_8192_tflops=round(f["tflops"], 1), fp8_frac_4p5pf=round(f["tflops"] / 4500.0, 4))
    if "skinny" in secondary:
        fr = {k: v["frac_hbm"] for k, v in secondary["skinny"]["cells"].items()}
        summary.update(skinny_frac_hbm_min=min(fr.values()), skinny_frac_hbm_max=max(fr.values()),
                       skinny_worst_cell=min(fr, key=fr.get))
    if "epilogue" in secondary and "nvfp4_4096" in secondary["epilogue"]["shapes"]:
        c2 = secondary["epilogue"]["shapes"]["nvfp4_4096"]
        summary.update(nvfp4_4096_graph_us=c2["plain"]["us"], nvfp4_4096_graph_us_pdl=c2["plain_pdl"]["us"])
    if "swizzle" in secondary:
        summary["swizzle_frac_hbm"] = secondary["swizzle"]["frac_hbm"]
    if "grouped" in secondary:
        summary["moe_frac_hbm"] = secondary["grouped"]["variants"]["scatter"]["frac_hbm"]
    if "packed" in secondary and "us" in secondary["packed"]:
        pu = secondary["packed"]["us"]
        summary.update(packed_gemm_graph_us=pu["packed"], row_major_gemm_graph_us=pu["tensor_map"],
                       packed_frac_9pf=round(w.flops / (pu["packed"] * 1e-6) / 1e12 / 9000.0, 4))
    if e2e is not None:
        summary.update(e2e_tflops=round(e2e["value"], 1),
                       e2e_frac_of_copy_bound=e2e["host_link"]["frac_of_copy_bound"])
    line["summary"] = summary
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, dist: Dist) -> None:
    """The oracle timed on the host cores: each step is a bounded sample of the
    workload (whole output rows), sized so the run ends in minutes."""
    if dist.rank != 0:
        return
    import oracle
    w = workloads.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    p = workloads.make_nvfp4(w, dev)
    host = {k: (p[k].cpu().numpy() if torch.is_tensor(p[k]) else p[k]) for k in ("A", "sfA", "B", "sfB")}
    o = oracle.get()
    threads = oracle.default_threads()
    per_step_rows = max(threads, 2 * threads)
    budget = max(5.0, 120.0 / max(1, args.steps + args.warmup))
    t = time.perf_counter()
    o.nvfp4_gemm(host["A"], host["sfA"], host["B"], host["sfB"], p["alpha"], w.K, rows=[0], nthreads=1)
    one_row_1t = time.perf_counter() - t
    per_step_rows = max(1, min(per_step_rows, int(budget * threads / max(one_row_1t, 1e-3))))
    times = []
    for i in range(args.warmup + args.steps):
        sel = [(i * per_step_rows + r) % w.M for r in range(per_step_rows)]
        t = time.perf_counter()
        o.nvfp4_gemm(host["A"], host["sfA"], host["B"], host["sfB"], p["alpha"], w.K, rows=sel,
                     nthreads=threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    ms = statistics.mean(times) * 1e3
    flops = 2.0 * per_step_rows * w.N * w.K
    value = flops / (ms * 1e-3) / 1e12
    sample = f"{per_step_rows} of {w.M} output rows x all {w.N} columns per step, K={w.K}"
    print(json.dumps({
        "metric": "NVFP4 GEMM TFLOPS at 16384^3 (whole hot path: scale prep + persistent GEMM)",
        "value": value, "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "cpu": host_cpu()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_case(args) -> None:
    """One GEMM shape alone (--case nvfp4:MxNxK, fp8:MxNxK, dense:MxNxK or
    densef16:MxNxK for NVFP4 x dense BF16 / FP16, packed:MxNxK for NVFP4 with tile-packed operands,
    optionally a forced --plan), the NVFP4 quantiser on BF16 ROWSxK (--case
    quantize:ROWSxK), or a grouped workload (--case grouped:NAME, e.g.
    grouped:moe_e64_t1024_k8; groupeddense:NAME for BF16 expert weights): `warmup` untimed then `steps` timed launches,
    inputs resident. Used for profiler captures of a single kernel and for ad-hoc
    timings; prints one JSON line."""
    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_precision_persistent_gb300 as bsg
    kind, shape = args.case.split(":")
    dims = [] if kind in ("grouped", "groupeddense") else [int(x) for x in shape.lower().split("x")]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.current_stream()
    bsg.bsg_set_raster_group(args.raster)
    if kind == "quantize":
        rows, K = dims
        g = torch.Generator(device="cpu").manual_seed(0xB5C0)
        x = torch.randn((rows, K), generator=g).to(torch.bfloat16).to(dev)
        packed = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
        swz = torch.empty(bsg.nvfp4_swizzled_scale_bytes(rows, K), dtype=torch.uint8, device=dev)
        gl = torch.empty(2, dtype=torch.float32, device=dev)
        for _ in range(args.warmup):
            bsg.nvfp4_quantize(rows, K, x, packed, swz, None, gl, s)
        torch.cuda.synchronize()
        evs = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            bsg.nvfp4_quantize(rows, K, x, packed, swz, None, gl, s)
            b.record(s)
            evs.append((a, b))
        torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
        moved = 2 * (2 * rows * K) + rows * K // 2 + bsg.nvfp4_swizzled_scale_bytes(rows, K)
        print(json.dumps({"case": args.case, "us": round(us, 2), "gb_s": round(moved / (us * 1e-6) / 1e9, 1)}),
              flush=True)
        return
    if kind in ("grouped", "groupeddense"):
        w = workloads.GROUPED_WORKLOADS[shape]
        if kind == "grouped":
            g = GroupedProblem(w, dev)
            moved = w.algorithmic_bytes
        else:
            # the routed GEMM with BF16 expert weights, D in token order
            offs, dst = workloads.routing(w.E, w.tokens, w.top_k, seed=1)
            offs, dst = offs.to(dev), dst.to(dev)
            pd = workloads.make_dense_grouped(w.E, w.M, w.N, w.K, seed=1, device=dev)
            sa = torch.empty(bsg.nvfp4_grouped_scale_bytes(w.E, w.M, w.K), dtype=torch.uint8, device=dev)
            bsg.nvfp4_swizzle_scales_grouped(w.E, w.M, w.K, offs, pd["sfA"], sa, s)
            Dg = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
            moved = w.M * w.K * 9 // 16 + w.E * w.N * w.K * 2 + w.M * w.N * 2

            def g():
                bsg.nvfp4_dense_grouped_gemm(w.E, w.M, w.N, w.K, pd["A"], sa, pd["B"], offs, pd["alpha"], None, None,
                                             dst, w.M, Dg, s)
        bsg.bsg_force_plan(args.plan)
        try:
            for _ in range(args.warmup):
                g()
            torch.cuda.synchronize()
            evs = []
            for _ in range(args.steps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                g()
                b.record(s)
                evs.append((a, b))
            torch.cuda.synchronize()
        finally:
            bsg.bsg_force_plan(None)
        if bsg.bsg_get_device_status() != bsg.BSG_OK:
            raise SystemExit("device status reported an error")
        us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
        print(json.dumps({"case": args.case, "plan": bsg.bsg_last_plan_name(), "us": round(us, 2),
                          "gb_s": round(moved / (us * 1e-6) / 1e9, 1)}), flush=True)
        return
    M, N, K = dims
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if kind == "nvfp4":
        p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], dev, M=M, N=N, K=K)
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, p["sfA"], sa, s)
        bsg.nvfp4_swizzle_scales(N, K, p["sfB"], sb, s)

        epi = set(args.epi.split(",")) if args.epi else set()
        e = workloads.make_epilogue(M, N, seed=3, bias_std=float(K) ** 0.5, device=dev)
        eb, eg, es = (e[k] if k in epi else None for k in ("bias", "gamma", "scatter"))

        def call():
            bsg.nvfp4_gemm_ex(M, N, K, p["A"], sa, p["B"], sb, p["alpha"], eb, eg, es, M, D, s)
    elif kind == "packed":
        # A and B packed into 16 KiB tiles once, outside the timed launches
        p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], dev, M=M, N=N, K=K)
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, p["sfA"], sa, s)
        bsg.nvfp4_swizzle_scales(N, K, p["sfB"], sb, s)
        ap = torch.empty(bsg.nvfp4_packed_operand_bytes(M, K), dtype=torch.uint8, device=dev)
        bp = torch.empty(bsg.nvfp4_packed_operand_bytes(N, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_pack_operand(M, K, p["A"], ap, s)
        bsg.nvfp4_pack_operand(N, K, p["B"], bp, s)

        def call():
            bsg.nvfp4_gemm_packed(M, N, K, ap, sa, bp, sb, p["alpha"], D, s)
    elif kind in ("dense", "densef16"):
        f16 = kind == "densef16"
        pd = workloads.make_dense(M, N, K, seed=1, device=dev, b_dtype=torch.float16 if f16 else torch.bfloat16)
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, pd["sfA"], sa, s)
        dense = bsg.nvfp4_dense_f16_gemm if f16 else bsg.nvfp4_dense_gemm

        def call():
            dense(M, N, K, pd["A"], sa, pd["B"], pd["alpha"], None, None, None, M, D, s)
    elif kind == "fp8":
        q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], dev, M=M, N=N, K=K)

        def call():
            bsg.fp8_gemm(M, N, K, q["A"], None, q["B"], None, q["alpha"], D, s)
    else:
        raise SystemExit(f"unknown case kind {kind!r}")
    bsg.bsg_force_plan(args.plan)
    try:
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        evs = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            call()
            b.record(s)
            evs.append((a, b))
        torch.cuda.synchronize()
        plan = bsg.bsg_last_plan_name()
    finally:
        bsg.bsg_force_plan(None)
    if bsg.bsg_get_device_status() != bsg.BSG_OK:
        raise SystemExit("device status reported an error")
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    print(json.dumps({"case": args.case, "plan": plan, "raster": args.raster or 16, "ms": round(ms, 5),
                      "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 2)}), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="nvfp4_16384",
                    choices=[n for n, w in workloads.WORKLOADS.items() if w.kind == "nvfp4"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--cpu-configs", action="store_true",
                    help="also time the oracle on every output of the smaller configurations")
    ap.add_argument("--case", default=None,
                    help="time one shape alone instead of the benchmark: nvfp4:MxNxK, fp8:MxNxK or "
                         "quantize:ROWSxK")
    ap.add_argument("--plan", default=None, help="with --case: force this plan")
    ap.add_argument("--raster", type=int, default=0,
                    help="with --case: M tiles per rasterisation group (0: the library default)")
    ap.add_argument("--epi", default=None,
                    help="with --case nvfp4: fused epilogue options, comma list of bias,gamma,scatter")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    dist = Dist(args.gpus) if args.impl == "ours" or args.gpus > 1 else Dist(1)
    try:
        if args.impl == "ours":
            run_ours(args, dist)
        else:
            run_reference(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
