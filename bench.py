#!/usr/bin/env python3
"""Benchmark libtgemm: FP16 GEMM TFLOP/s and fraction of the tensor roofline
on the transformer-MLP workload (8192×28672×4096, fused ReLU), with the
skinny weight-streaming workload (64×16384×8192) measured beside it in HBM
GB/s.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one tg_gemm_f16 launch over one batch of synthetic input (the whole
hot path: tensor maps, persistent tile schedule, TMA ring, tcgen05 MMA into
TMEM, fused ReLU + fp16 epilogue with TMA stores).  Inputs are larger than L2,
so no flush is needed between steps.  Every leg times its launches back to
back between two CUDA events on the launching stream (no event between
launches) and divides by their number; 20 further launches, each between its
own events, give the min / median of an isolated launch as context.  N > 1
runs N independent replicas (one
per GPU, no collective on the data path); value = work of all ranks ÷ the
slowest rank's time.

--impl reference times the CPU oracle (oracle/) as it stands on this host's
cores, on a bounded row slab of the same workload per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP16 GEMM TFLOP/s and % of dense tensor peak (HBM GB/s % for skinny M), 1 GB300"
MAIN_WORKLOAD = "mlp_8192x28672x4096_relu"
SKINNY_WORKLOAD = "skinny_64x16384x8192"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def parse_args(argv=None):
    from tiled_fp16_gemm_gb300 import workloads as W
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=MAIN_WORKLOAD)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-skinny", action="store_true")
    p.add_argument("--no-bf16", action="store_true")
    p.add_argument("--no-epilogue", action="store_true")
    p.add_argument("--no-mxfp4", action="store_true")
    p.add_argument("--no-sp24", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the 256^3, 1024^3 ReLU and 4096^3 configs and the staged layout")
    p.add_argument("--no-library", action="store_true",
                   help="skip the cuBLAS (torch.matmul) context timings")
    p.add_argument("--sp24-workload", default="sp24_mlp_8192x28672x4096_relu",
                   choices=sorted(W.SP24_WORKLOADS))
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    return a


# ------------------------------------------------------------------ helpers

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def source_hash(files=None) -> str:
    """Hash of kernel sources (the given csrc file names, else all of csrc),
    to tell whether stored ncu counters are stale."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_fp16_gemm_gb300", "csrc")
    for name in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def load_peaks():
    """(HBM copy GB/s, dense bf16 TFLOP/s burst, the same sustained under the
    power cap, "measured" | "fallback")."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        burst = float(d["bf16_tflops"])
        return (float(d["hbm_gbs"]), burst, float(d.get("bf16_tflops_sustained", burst)),
                "measured")
    except Exception:
        return (FALLBACK_PEAKS["hbm_gbs"], FALLBACK_PEAKS["bf16_tflops"],
                FALLBACK_PEAKS["bf16_tflops_sustained"], "fallback")


def tensor_roofline(achieved, clk, peaks, scale=1.0, what="dense bf16"):
    """Roofline of a tensor-bound leg.  The denominator is the measured burst
    rate, or the measured sustained rate where the leg's own clock record shows
    the power cap active (the kernel ran inside a long, power-capped run); the
    fraction of the burst rate is given as well.  scale: 2 for the 2:4 sparse
    rate (the nominal sparse-to-dense ratio)."""
    _, burst, sustained, src = peaks
    capped = bool(clk) and "sw_power_cap" in (clk.get("reasons") or [])
    peak = scale * (sustained if capped else burst)
    kind = ("sustained (this leg ran under sw_power_cap)" if capped else "burst")
    pre = f"{scale:g} x " if scale != 1.0 else ""
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "frac_of_burst": achieved / (scale * burst),
            "peak_source": f"{pre}{src} {what} {kind}"}


def stored_traffic(kernel_key: str):
    """dram bytes per launch from a committed ncu capture, if taken on the
    current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_hash") == source_hash(e.get("sources")):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while work runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 100):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.5)  # let the sampler come up before the timed region

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[5:]))
                except Exception:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:  # timed region shorter than one period: nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4][1:5])
                          if v.lower() == "active"})
        return {
            "sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
            "sm_max_mhz": max(r[2] for r in inside) if inside else None,
            "power_w_max": max(r[3] for r in inside) if inside else None,
            "samples": len(inside),
            "reasons": reasons,
        }


class NvmlSampler:
    """SM clock, power and clock-event reasons of this process's GPU, read
    through NVML (libnvidia-ml, ctypes) every `period_s` seconds on a thread
    while work runs.  Reads only; changes no setting.  The GPU is found by its
    PCI bus id, so the NVML index need not match the CUDA one."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device, period_s: float = 0.005):
        import ctypes
        import threading
        self.period_s = period_s
        self.samples = []
        self._stop = threading.Event()
        self._thread = None
        self.ok = False
        try:
            import torch
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            pr = torch.cuda.get_device_properties(device)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # 1: SM clock
                return
            self.lib, self.h, self.max_mhz = lib, h, int(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        import ctypes
        mhz, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.time()
            a = self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
            b = self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw))
            c = self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs))
            if a == 0:
                self.samples.append((t, int(mhz.value), mw.value / 1e3 if b == 0 else None,
                                     int(rs.value) if c == 0 else 0))
            time.sleep(self.period_s)

    def start(self):
        import threading
        if not self.ok:
            return
        self.samples = []
        self._stop.clear()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        if self.ok and self._thread is not None:
            self._stop.set()
            self._thread.join()

    def window(self, t0: float, t1: float):
        """Summary of the samples taken between wall times t0 and t1."""
        if not self.ok:
            return None
        inside = [r for r in list(self.samples) if t0 <= r[0] <= t1]
        if not inside:
            return None
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items()
                          if r[3] & bit})
        pw = [r[2] for r in inside if r[2] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_mhz_min": min(r[1] for r in inside), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(pw) if pw else None, "samples": len(inside),
                "reasons": reasons, "source": f"NVML every {self.period_s * 1e3:.0f} ms"}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ timing

PER_LAUNCH_SAMPLES = 20
_NVML = None             # NvmlSampler running through the whole bench, if NVML loads
LAST_LEG_CLOCKS = None   # its summary over the last timed region


# Idle time before each timed leg, so that a leg starts from an idle GPU as
# the first one does and does not inherit the power state (clock cap) that
# the legs before it left.
LEG_IDLE_S = 1.0
LEG_REWARM = 3  # launches between the idle and the timed region


def time_launches(launch, stream, steps: int, world: int, device):
    """Time `steps` back-to-back launches on `stream` between two CUDA events,
    with no event between launches: consecutive launches overlap their
    start-up with the previous launch's tail, as in any stream of kernels.
    The leg starts after LEG_IDLE_S of idle and LEG_REWARM untimed launches.
    Returns (total_ms, mean_ms = total_ms / steps, per_ms, wall0, wall1).
    per_ms holds PER_LAUNCH_SAMPLES further launches, each bracketed by its
    own events; those events serialise the launches, so per_ms is context
    (min / median of an isolated launch), not the throughput."""
    import torch
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    time.sleep(LEG_IDLE_S)
    for _ in range(LEG_REWARM):  # clocks back up after the idle
        launch()
    barrier(world, device)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_begin.record(stream)
    for _ in range(steps):
        launch()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world, device)
    wall1 = time.time()
    total = t_begin.elapsed_time(t_end)
    global LAST_LEG_CLOCKS
    LAST_LEG_CLOCKS = _NVML.window(wall0, wall1) if _NVML is not None else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(PER_LAUNCH_SAMPLES)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(PER_LAUNCH_SAMPLES)]
    for i in range(PER_LAUNCH_SAMPLES):
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total, total / steps, per, wall0, wall1


def interleaved_times(launch_a, launch_b, stream, block: int, rounds: int):
    """Mean ms per launch of `launch_a` and of `launch_b`, from blocks of `block`
    back-to-back launches of each taken in turn (`rounds` of each, each block
    between its own two events), so both see the same clocks and temperature."""
    import torch
    ta = tb = 0.0
    for _ in range(rounds):
        for fn, which in ((launch_a, 0), (launch_b, 1)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(block):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if which == 0:
                ta += e0.elapsed_time(e1)
            else:
                tb += e0.elapsed_time(e1)
    return ta / (block * rounds), tb / (block * rounds)


def interleaved_ratio(launch_a, launch_b, stream, block: int, rounds: int) -> float:
    """Time of `launch_a` over time of `launch_b` (interleaved_times)."""
    ta, tb = interleaved_times(launch_a, launch_b, stream, block, rounds)
    return ta / tb


def library_context(launch_on, a_sets, b_sets, stream, flops: float, relu: bool,
                    min_bytes: float = 0.0):
    """The same product through torch.matmul (cuBLAS, fp16, no epilogue) on the
    same operand copies.  Both sides are captured in CUDA graphs of `block`
    launches each (this library's through launch_on(stream handle), on a
    stream that ran it once before capture), and the two graphs are replayed
    in turn, so neither side's host dispatch hides its kernel time at small
    sizes.  Context only: nothing of the library's path calls cuBLAS."""
    import torch
    sets = len(a_sets)
    outs = [torch.empty((a_sets[0].shape[0], b_sets[0].shape[1]), dtype=torch.float16,
                        device=a_sets[0].device) for _ in range(sets)]
    one = flops / 1.8e15 * 1e3  # ms per launch, roughly
    block = int(max(3, min(200, 5.0 / max(one, 1e-4))))
    cs = torch.cuda.Stream(a_sets[0].device)
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        for j in range(3):
            launch_on(cs.cuda_stream)
            torch.matmul(a_sets[j % sets], b_sets[j % sets], out=outs[j % sets])
    torch.cuda.synchronize()
    g_ours, g_lib = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ours, stream=cs):
        for _ in range(block):
            launch_on(cs.cuda_stream)
    with torch.cuda.graph(g_lib, stream=cs):
        for j in range(block):
            torch.matmul(a_sets[j % sets], b_sets[j % sets], out=outs[j % sets])
    torch.cuda.synchronize()
    t = [0.0, 0.0]
    rounds = 4
    with torch.cuda.stream(stream):
        g_ours.replay()
        g_lib.replay()
        torch.cuda.synchronize()
        for _ in range(rounds):
            for which, g in ((0, g_ours), (1, g_lib)):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                t[which] += e0.elapsed_time(e1)
    ours, lib = t[0] / (block * rounds), t[1] / (block * rounds)
    del g_ours, g_lib, outs
    r = {"call": "torch.matmul (cuBLAS), fp16" + (", without the ReLU" if relu else ""),
         "ms_mean": lib, "tflops": flops / (lib / 1e3) / 1e12,
         "ours_ms_mean_graph": ours, "ours_over_library_time": ours / lib,
         "how": f"each side a CUDA graph of {block} launches; 4 replays of each, in turn"}
    if min_bytes:
        r["gbs"] = min_bytes / (lib / 1e3) / 1e9
    return r


def rotating_sets(set_bytes: int) -> int:
    """Copies of one problem's operands to rotate through so that the copies
    together span at least twice L2: each launch then reads operands that
    the launches before it have evicted."""
    return int(min(1024, max(1, -(-2 * L2_BYTES // max(set_bytes, 1)))))


def host_issue_us(launch, n: int) -> float:
    """Host time per call to enqueue `n` launches (no synchronisation inside)."""
    import torch
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(n):
        launch()
    dt = time.perf_counter() - t
    torch.cuda.synchronize()
    return dt / n * 1e6


def link_bound(h2d_bytes: int, d2h_bytes: int, device):
    """Pinned host <-> device copy rates measured now, alone and with both
    directions at once, and the shortest time in which a step can move its
    bytes: no end-to-end step can be faster than its concurrent copies."""
    import torch
    hu = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    du = torch.empty(h2d_bytes, dtype=torch.uint8, device=device)
    hd = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    dd = torch.empty(d2h_bytes, dtype=torch.uint8, device=device)
    s_up, s_down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    cur = torch.cuda.current_stream(device)

    def timed(up: bool, down: bool) -> float:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(cur)
        s_up.wait_event(ev[0])
        s_down.wait_event(ev[0])
        if up:
            with torch.cuda.stream(s_up):
                du.copy_(hu, non_blocking=True)
        if down:
            with torch.cuda.stream(s_down):
                hd.copy_(dd, non_blocking=True)
        ev[1].record(s_up)
        ev[2].record(s_down)
        torch.cuda.synchronize()
        return max(ev[0].elapsed_time(ev[1]), ev[0].elapsed_time(ev[2]))

    best = {}
    for key, up, down in (("up", True, False), ("down", False, True), ("both", True, True)):
        timed(up, down)
        best[key] = min(timed(up, down) for _ in range(3))
    del hu, du, hd, dd
    return {
        "h2d_gbs_alone": h2d_bytes / (best["up"] / 1e3) / 1e9,
        "d2h_gbs_alone": d2h_bytes / (best["down"] / 1e3) / 1e9,
        "both_directions_ms": best["both"],
        "how": "contiguous pinned copies of the step's bytes on two streams, best of 3",
    }


def cpu_oracle_rate(A, B, w, seconds: float):
    """Time the oracle on a row slab sized for about `seconds` of work.
    Returns (tflops, rows, elapsed_s, threads)."""
    import oracle
    o = oracle.default()
    th = o.num_threads()
    rows = max(1, min(w.M, th))
    t = time.perf_counter()
    o.gemm(A[:rows], B, rows, w.N, w.K, relu=w.relu)
    dt = time.perf_counter() - t
    rows2 = int(max(rows, min(w.M, rows * seconds / max(dt, 1e-6))))
    t = time.perf_counter()
    o.gemm(A[:rows2], B, rows2, w.N, w.K, relu=w.relu)
    dt2 = time.perf_counter() - t
    return 2.0 * rows2 * w.N * w.K / dt2 / 1e12, rows2, dt2, th


# ------------------------------------------------------------------ arms

def run_reference(args, w):
    """The CPU oracle as it stands, timed on this host's cores."""
    import oracle
    from tiled_fp16_gemm_gb300 import workloads as W
    A, B = W.workload_inputs(w)
    o = oracle.default()
    th = o.num_threads()
    rows = max(1, min(w.M, th))
    t = time.perf_counter()
    o.gemm(A[:rows], B, rows, w.N, w.K, relu=w.relu)
    per_row = (time.perf_counter() - t) / rows
    budget = 150.0 / (args.steps + args.warmup)
    rows = int(max(1, min(w.M, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        o.gemm(A[:rows], B, rows, w.N, w.K, relu=w.relu)
    t = time.perf_counter()
    for _ in range(args.steps):
        o.gemm(A[:rows], B, rows, w.N, w.K, relu=w.relu)
    dt = time.perf_counter() - t
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / dt / 1e12
    sample = f"{rows} of {w.M} rows of {w.name} per step (full N and K)"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def config_block(w, gpus):
    inb = 2 * (w.M * w.K + w.K * w.N)
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
            "epilogue": "relu" if w.relu else "none",
            "inputs": f"A {w.dist_a}, B {w.dist_b}, seed {w.seed}",
            "l2": (f"inputs larger than L2 ({inb / 2**20:.0f} MiB of A+B vs "
                   f"{L2_BYTES // 2**20} MiB L2); no flush" if inb > L2_BYTES else
                   f"inputs fit in L2 ({inb / 2**20:.0f} MiB of A+B vs {L2_BYTES // 2**20} MiB "
                   "L2) and stay there between launches"),
            "parallelism": "replicas" if gpus > 1 else "single GPU"}


def time_config(tg, w, args, stream, world, device, nsm, peaks):
    """One of the square configs through tg_gemm_f16, timed like the main
    workload (back-to-back launches between two events), its operands rotated
    over copies spanning twice L2."""
    import torch
    from tiled_fp16_gemm_gb300 import workloads as W
    A, B = W.workload_inputs(w)
    sets = rotating_sets(w.min_bytes)
    a = torch.from_numpy(A).to(device).unsqueeze(0).repeat(sets, 1, 1)
    b = torch.from_numpy(B).to(device).unsqueeze(0).repeat(sets, 1, 1)
    c = torch.empty((sets, w.M, w.N), dtype=torch.float16, device=device)
    epi = tg.TG_EPI_RELU if w.relu else tg.TG_EPI_NONE
    plan = tg.tg_plan_f16(w.M, w.N, w.K, nsm)
    ptrs = [(a[i].data_ptr(), b[i].data_ptr(), c[i].data_ptr()) for i in range(sets)]
    ctr = [0]
    fn = tg.library().tg_gemm_f16
    sp = stream.cuda_stream

    def launch_on(sh):
        pa, pb, pc = ptrs[ctr[0] % sets]
        ctr[0] += 1
        st = fn(pa, pb, pc, w.M, w.N, w.K, w.K, w.N, w.N, epi, sh)
        if st != tg.TG_OK:
            raise tg.TgemmError(st)

    def launch():
        launch_on(sp)

    for _ in range(max(args.warmup, sets)):
        launch()
    tg.sync_status(stream)
    n = max(200, args.steps) if w.flops < 1e11 else max(100, args.steps // 2)
    _, k, per, _, _ = time_launches(launch, stream, n, world, device)
    tg.sync_status(stream)
    host_us = host_issue_us(launch, n)
    tg.sync_status(stream)
    lib = None
    if not args.no_library:
        lib = library_context(launch_on, [a[i] for i in range(sets)],
                              [b[i] for i in range(sets)], stream, float(w.flops), w.relu)
        tg.sync_status(stream)
    tf = w.flops / (k / 1e3) / 1e12
    if plan.cluster == 2:
        kname = (f"tg_gemm_f16_pair<{plan.stages} stages of {plan.bk} k>, last wave in "
                 f"{plan.split_k} k-pieces x {plan.split_n} column pieces per tile")
    else:
        kname = f"tg_gemm_f16_persistent<{plan.bn},{plan.stages}>"
    del a, b, c
    torch.cuda.empty_cache()
    return {
        "workload": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": "relu" if w.relu else "none",
        "kernel": kname, "grid": int(plan.grid), "tiles": int(plan.num_tiles),
        "launches": n, "operand_sets": sets,
        "l2": f"operands rotated over {sets} copies ({sets * w.min_bytes / 2**20:.0f} MiB)",
        "kernel_ms_mean": k, "isolated_launch_ms_min": min(per), "clocks": LAST_LEG_CLOCKS,
        "isolated_launch_ms_median": statistics.median(per),
        "host_us_per_call": host_us,
        "tflops": tf, "gbs": w.min_bytes / (k / 1e3) / 1e9,
        "roofline": tensor_roofline(tf, LAST_LEG_CLOCKS, peaks),
        "library_context": lib,
    }


def run_ours(args, w, rank, world, local_rank):
    import numpy as np
    import torch
    import tiled_fp16_gemm_gb300 as tg
    from tiled_fp16_gemm_gb300 import workloads as W

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    nsm = torch.cuda.get_device_properties(device).multi_processor_count
    peaks = load_peaks()
    hbm_peak, _, _, peak_src = peaks

    A, B = W.workload_inputs(w)
    a = torch.from_numpy(A).to(device)
    b = torch.from_numpy(B).to(device)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=device)
    epi = tg.TG_EPI_RELU if w.relu else tg.TG_EPI_NONE
    plan = tg.tg_plan_f16(w.M, w.N, w.K, nsm)

    def launch_on(sh):
        st = tg.tg_gemm_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), w.M, w.N, w.K, w.K, w.N,
                            w.N, epi, sh)
        if st != tg.TG_OK:
            raise tg.TgemmError(st)

    def launch():
        launch_on(stream.cuda_stream)

    for _ in range(args.warmup):
        launch()
    tg.sync_status(stream)

    global _NVML
    _NVML = NvmlSampler(device)
    clocks = None if _NVML.ok else ClockSampler(local_rank)
    if _NVML.ok:
        _NVML.start()
    else:
        clocks.start()
    total_ms, _, per, wall0, wall1 = time_launches(launch, stream, args.steps, world, device)
    clk = _NVML.window(wall0, wall1) if _NVML.ok else None
    if clk is None:
        clk = clocks.stop(wall0, wall1) if clocks is not None else {
            "sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"]}
    tg.sync_status(stream)
    total_ms = max_over_ranks(total_ms, world, device)

    flops = float(w.flops)
    ms_step = total_ms / args.steps
    value = world * flops * args.steps / (total_ms / 1e3) / 1e12
    kernel_ms = ms_step
    achieved = flops / (kernel_ms / 1e3) / 1e12
    if plan.kernel == tg.TG_KERNEL_PERSISTENT:
        if plan.cluster == 2:
            kernel_key = "pair256"
            kname = (f"tg_gemm_f16_pair<{plan.stages} stages of {plan.bk} k> "
                     "(CTA pairs, 256x256 tiles)")
        else:
            kernel_key = f"persistent_bn{plan.bn}"
            kname = f"tg_gemm_f16_persistent<{plan.bn},{plan.stages}>"
        roof = tensor_roofline(achieved, clk, peaks)
    else:  # skinny split-K: bound by streaming B from HBM
        kernel_key = "skinny"
        kname = "tg_gemm_f16_skinny"
        gbs = w.min_bytes / (kernel_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbs / hbm_peak, "peak_source": f"{peak_src} copy bandwidth"}
    roof["traffic"] = stored_traffic(f"{kernel_key}:{w.name}")
    roof.update({"kernel": kname, "kernel_ms_mean": kernel_ms,
                 "isolated_launch_ms_min": min(per),
                 "isolated_launch_ms_median": statistics.median(per)})
    lib_ctx = None
    if not args.no_library:
        lib_ctx = library_context(launch_on, [a], [b], stream, float(w.flops), w.relu)
        tg.sync_status(stream)
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic", "config": config_block(w, world),
        "roofline": roof,
        "gpu_launches": args.steps,
        "clocks": clk,
        "leg_idle_s": LEG_IDLE_S,
    }
    if lib_ctx is not None:
        out["library_context"] = lib_ctx

    # ---- the other square configs (256^3, 1024^3 with ReLU, 4096^3), same
    # method; operands rotate over enough copies that each launch reads them
    # from HBM, not from what the previous launch left in L2
    if not args.no_configs and w.name == MAIN_WORKLOAD:
        out["configs"] = {}
        for cname in ("gemm_256", "gemm_1024_relu", "gemm_4096"):
            out["configs"][cname] = time_config(tg, W.WORKLOADS[cname], args, stream, world,
                                                device, nsm, peaks)
        out["configs"][MAIN_WORKLOAD] = {"see": "top level (value, roofline)"}
        out["configs"][SKINNY_WORKLOAD] = {"see": "skinny"}

        # the main workload with A in a layout the tensor memory-access unit
        # cannot address (lda = K + 1): A is first copied to an aligned
        # staging buffer, then the same kernel runs
        a_odd = torch.zeros((w.M, w.K + 1), dtype=torch.float16, device=device)
        a_odd[:, :w.K] = a
        c_odd = torch.empty_like(c)

        def launch_odd():
            st = tg.tg_gemm_f16(a_odd.data_ptr(), b.data_ptr(), c_odd.data_ptr(), w.M, w.N, w.K,
                                w.K + 1, w.N, w.N, epi, stream.cuda_stream)
            if st != tg.TG_OK:
                raise tg.TgemmError(st)

        for _ in range(args.warmup):
            launch_odd()
        launch()
        tg.sync_status(stream)
        same = bool(torch.equal(c_odd.view(torch.int16), c.view(torch.int16)))
        n_odd = max(50, args.steps // 2)
        _, k_odd, per_odd, _, _ = time_launches(launch_odd, stream, n_odd, world, device)
        tg.sync_status(stream)
        out["staged_layout"] = {
            "workload": w.name, "lda": w.K + 1, "launches": n_odd,
            "what": "A copied to an aligned staging buffer (tg_copy_matrix16), then the "
                    "planned kernel",
            "kernel_ms_mean": k_odd, "isolated_launch_ms_min": min(per_odd),
            "clocks": LAST_LEG_CLOCKS,
            "tflops": flops / (k_odd / 1e3) / 1e12,
            "vs_aligned": kernel_ms / k_odd,
            "staging_bytes": 2 * 2 * w.M * w.K,
            "same_bits_as_aligned": same,
        }
        del a_odd, c_odd

    # ---- skinny weight-streaming workload, same method
    if not args.no_skinny and w.name != SKINNY_WORKLOAD:
        ws = W.WORKLOADS[SKINNY_WORKLOAD]
        As, Bs = W.workload_inputs(ws)
        a2 = torch.from_numpy(As).to(device)
        b2 = torch.from_numpy(Bs).to(device)
        c2 = torch.empty((ws.M, ws.N), dtype=torch.float16, device=device)

        def launch2_on(sh):
            st = tg.tg_gemm_f16(a2.data_ptr(), b2.data_ptr(), c2.data_ptr(), ws.M, ws.N, ws.K,
                                ws.K, ws.N, ws.N, 0, sh)
            if st != tg.TG_OK:
                raise tg.TgemmError(st)

        def launch2():
            launch2_on(stream.cuda_stream)

        for _ in range(args.warmup):
            launch2()
        tg.sync_status(stream)
        n2 = max(50, args.steps)
        _, k2, per2, _, _ = time_launches(launch2, stream, n2, world, device)
        tg.sync_status(stream)
        gbs = ws.min_bytes / (k2 / 1e3) / 1e9
        out["skinny"] = {
            "workload": ws.name, "launches": n2, "kernel_ms_mean": k2,
            "isolated_launch_ms_min": min(per2), "isolated_launch_ms_median": statistics.median(per2),
            "clocks": LAST_LEG_CLOCKS,
            "tflops": ws.flops / (k2 / 1e3) / 1e12,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak,
                         "traffic": stored_traffic(f"skinny:{ws.name}"),
                         "peak_source": f"{peak_src} copy bandwidth"},
        }
        if not args.no_library:
            out["skinny"]["library_context"] = library_context(
                launch2_on, [a2], [b2], stream, float(ws.flops), False, float(ws.min_bytes))
            tg.sync_status(stream)
        del a2, b2, c2

    # ---- bfloat16 variant on the same shape, same method
    if not args.no_bf16:
        ab = a.to(torch.bfloat16)
        bb = b.to(torch.bfloat16)
        cb = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)

        def launch3():
            st = tg.tg_gemm_bf16(ab.data_ptr(), bb.data_ptr(), cb.data_ptr(), w.M, w.N, w.K,
                                 w.K, w.N, w.N, epi, stream.cuda_stream)
            if st != tg.TG_OK:
                raise tg.TgemmError(st)

        for _ in range(args.warmup):
            launch3()
        tg.sync_status(stream)
        n4 = max(50, args.steps // 2)
        _, k4, per4, _, _ = time_launches(launch3, stream, n4, world, device)
        tg.sync_status(stream)
        if plan.kernel == tg.TG_KERNEL_PERSISTENT:
            ach = flops / (k4 / 1e3) / 1e12
            roof4 = tensor_roofline(ach, LAST_LEG_CLOCKS, peaks)
        else:
            ach = w.min_bytes / (k4 / 1e3) / 1e9
            roof4 = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                     "frac": ach / hbm_peak}
        out["bf16"] = {"workload": w.name, "entry": "tg_gemm_bf16", "launches": n4,
                       "kernel_ms_mean": k4, "isolated_launch_ms_min": min(per4),
                       "clocks": LAST_LEG_CLOCKS,
                       "tflops": flops / (k4 / 1e3) / 1e12, "roofline": roof4}
        del ab, bb, cb

    # ---- extended epilogue on the same shape: bias + ReLU + residual (16-bit
    # out) and bias + ReLU with fp32 out, through tg_gemm_ex, same method
    if not args.no_epilogue:
        rng = np.random.default_rng(w.seed + 101)
        bias = torch.from_numpy(rng.normal(0.0, 0.5, size=w.N).astype(np.float32)).to(device)
        resid = torch.empty((w.M, w.N), dtype=torch.float16, device=device).normal_()
        variants = {"bias_relu_residual_f16": (resid, tg.TG_DTYPE_F16, torch.float16),
                    "bias_relu_f32": (None, tg.TG_DTYPE_F32, torch.float32)}
        out["epilogue"] = {"workload": w.name, "entry": "tg_gemm_ex"}
        for name, (r, odt, tdt) in variants.items():
            ce = torch.empty((w.M, w.N), dtype=tdt, device=device)
            ex = tg.tg_epilogue_ex_t(epi, odt, bias.data_ptr(),
                                     r.data_ptr() if r is not None else None,
                                     w.N if r is not None else 0)

            def launch5(ce=ce, ex=ex):
                st = tg.tg_gemm_ex(tg.TG_DTYPE_F16, a.data_ptr(), b.data_ptr(), ce.data_ptr(),
                                   w.M, w.N, w.K, w.K, w.N, w.N, ex, stream.cuda_stream)
                if st != tg.TG_OK:
                    raise tg.TgemmError(st, "tg_gemm_ex")

            for _ in range(args.warmup):
                launch5()
            tg.sync_status(stream)
            n5 = max(50, args.steps // 2)
            _, k5, per5, _, _ = time_launches(launch5, stream, n5, world, device)
            tg.sync_status(stream)
            # bytes the epilogue adds: the residual read, the wider output
            extra = (w.M * w.N * 2 if r is not None else 0) + w.N * 4 + \
                (w.M * w.N * 2 if odt == tg.TG_DTYPE_F32 else 0)
            ent = {"launches": n5, "kernel_ms_mean": k5, "isolated_launch_ms_min": min(per5),
                   "clocks": LAST_LEG_CLOCKS,
                   "extra_bytes": extra, "vs_plain": kernel_ms / k5,
                   "vs_plain_interleaved": interleaved_ratio(launch, launch5, stream, 10, 5)}
            if plan.kernel == tg.TG_KERNEL_PERSISTENT:
                ach = flops / (k5 / 1e3) / 1e12
                ent["roofline"] = tensor_roofline(ach, LAST_LEG_CLOCKS, peaks)
            else:
                ach = (w.min_bytes + extra) / (k5 / 1e3) / 1e9
                ent["roofline"] = {"bound": "hbm", "achieved": ach, "peak": hbm_peak,
                                   "unit": "GB/s", "frac": ach / hbm_peak}
            out["epilogue"][name] = ent
            del ce
        del bias, resid

    # ---- MXFP4 weights (tg_gemm_mxfp4): weight streaming through the fused
    # split-K kernel, and the MLP shape through dequantise-then-GEMM
    if not args.no_mxfp4 and world == 1:
        out["mxfp4"] = {"entry": "tg_gemm_mxfp4"}
        for mname in ("mxfp4_skinny_64x16384x8192", "mxfp4_mlp_8192x28672x4096_relu"):
            mw = W.MX_WORKLOADS[mname]
            Am, Bqm, Sm = W.mx_workload_inputs(mw)
            am = torch.from_numpy(Am).to(device)
            bqm = torch.from_numpy(Bqm).to(device)
            sm = torch.from_numpy(Sm).to(device)
            cm = torch.empty((mw.M, mw.N), dtype=torch.float16, device=device)
            ex_m = tg.tg_epilogue_ex_t(tg.TG_EPI_RELU if mw.relu else tg.TG_EPI_NONE,
                                       tg.TG_DTYPE_F16, None, None, 0)

            def launch6(am=am, bqm=bqm, sm=sm, cm=cm, mw=mw, ex_m=ex_m):
                st = tg.tg_gemm_mxfp4(am.data_ptr(), bqm.data_ptr(), sm.data_ptr(), cm.data_ptr(),
                                      mw.M, mw.N, mw.K, mw.K, bqm.shape[1], sm.shape[1], mw.N,
                                      ex_m, stream.cuda_stream)
                if st != tg.TG_OK:
                    raise tg.TgemmError(st, "tg_gemm_mxfp4")

            for _ in range(args.warmup):
                launch6()
            tg.sync_status(stream)
            n6 = max(50, args.steps // 2) if mw.M <= 128 else max(20, args.steps // 10)
            _, k6, per6, _, _ = time_launches(launch6, stream, n6, world, device)
            tg.sync_status(stream)
            ent = {"workload": mname, "launches": n6, "kernel_ms_mean": k6,
                   "isolated_launch_ms_min": min(per6), "tflops": mw.flops / (k6 / 1e3) / 1e12,
                   "clocks": LAST_LEG_CLOCKS}
            if mw.M <= 128:
                gbs = mw.min_bytes / (k6 / 1e3) / 1e9
                ent["kernel"] = "tg_gemm_mxfp4_skinny (codes decoded by converter warps into tensor memory)"
                ent["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                                   "unit": "GB/s", "frac": gbs / hbm_peak,
                                   "traffic": stored_traffic(f"mxfp4_skinny:{mname}"),
                                   "peak_source": f"{peak_src} copy bandwidth"}
                if "skinny" in out:
                    ent["vs_fp16_skinny"] = out["skinny"]["kernel_ms_mean"] / k6
            else:
                tf = mw.flops / (k6 / 1e3) / 1e12
                ent["kernel"] = "tg_mxfp4_dequant_f16 + tg_gemm_f16_pair (256x256 tiles)"
                ent["roofline"] = tensor_roofline(tf, LAST_LEG_CLOCKS, peaks)
            out["mxfp4"][mname] = ent
            del am, bqm, sm, cm

    # ---- 2:4 structured-sparse A (tg_gemm_sp24) on the MLP shape
    if not args.no_sp24 and world == 1:
        sw = W.SP24_WORKLOADS[args.sp24_workload]
        Acs, Es, Bs = W.sp24_workload_inputs(sw)
        acs = torch.from_numpy(Acs).to(device)
        es = torch.from_numpy(Es.view(np.int32)).to(device)
        bs = torch.from_numpy(Bs).to(device)
        cs = torch.empty((sw.M, sw.N), dtype=torch.float16, device=device)
        ex_s = tg.tg_epilogue_ex_t(tg.TG_EPI_RELU if sw.relu else tg.TG_EPI_NONE,
                                   tg.TG_DTYPE_F16, None, None, 0)

        def launch7():
            st = tg.tg_gemm_sp24(tg.TG_DTYPE_F16, acs.data_ptr(), es.data_ptr(), bs.data_ptr(),
                                 cs.data_ptr(), sw.M, sw.N, sw.K, sw.K // 2, sw.K // 32, sw.N,
                                 sw.N, ex_s, stream.cuda_stream)
            if st != tg.TG_OK:
                raise tg.TgemmError(st, "tg_gemm_sp24")

        def time_sp24(force):
            """Mean / min ms of launch7 with TGEMM_FORCE_SP24 = force (None: the
            library's own choice, the CTA-pair kernel at this shape)."""
            prev = os.environ.pop("TGEMM_FORCE_SP24", None)
            if force is not None:
                os.environ["TGEMM_FORCE_SP24"] = force
            try:
                for _ in range(args.warmup):
                    launch7()
                tg.sync_status(stream)
                _, mean, per, _, _ = time_launches(launch7, stream, n7, world, device)
                sp_clocks[force] = LAST_LEG_CLOCKS
                tg.sync_status(stream)
            finally:
                os.environ.pop("TGEMM_FORCE_SP24", None)
                if prev is not None:
                    os.environ["TGEMM_FORCE_SP24"] = prev
            return mean, min(per)

        n7 = max(20, args.steps // 10)
        sp_clocks = {}
        k7, min7 = time_sp24(None)
        k7c, min7c = time_sp24("cta")
        tf7 = sw.flops / (k7 / 1e3) / 1e12
        out["sp24"] = {
            "workload": sw.name, "entry": "tg_gemm_sp24", "launches": n7,
            "kernel": "tg_gemm_sp24_pair<4, __half, false> (tcgen05.mma.sp cta_group::2, "
                      "256x256 tiles, 4 stages: the plain-epilogue build)",
            "kernel_ms_mean": k7, "isolated_launch_ms_min": min7, "clocks": sp_clocks.get(None),
            "tflops_dense_equivalent": tf7,
            "vs_dense_pair": kernel_ms / k7 if (sw.M, sw.N, sw.K) == (w.M, w.N, w.K) else None,
            "roofline": dict(tensor_roofline(tf7, sp_clocks.get(None), peaks, scale=2.0),
                             traffic=stored_traffic(f"sp24_pair:{sw.name}")),
            "one_cta_kernel": {
                "kernel": "tg_gemm_sp24 (tcgen05.mma.sp, 128x128 tiles)", "launches": n7,
                "kernel_ms_mean": k7c, "isolated_launch_ms_min": min7c,
                "tflops_dense_equivalent": sw.flops / (k7c / 1e3) / 1e12,
                "traffic": stored_traffic(f"sp24:{sw.name}")},
        }
        del acs, es, bs, cs

    # ---- end to end through the public API, host buffers in and out
    if not args.no_e2e:
        ha = torch.from_numpy(A).pin_memory()
        hb = torch.from_numpy(B).pin_memory()
        n3 = max(5, min(args.steps, 20))
        tg.gemm_host(ha, hb, relu=w.relu, stream=stream)  # warm
        barrier(world, device)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(n3):
            tg.gemm_host(ha, hb, relu=w.relu, stream=stream)
        dt = max_over_ranks(time.perf_counter() - t, world, device)
        e2e_value = world * flops * n3 / dt / 1e12
        h2d = int(ha.numel() * 2 + hb.numel() * 2)
        d2h = int(w.M * w.N * 2)
        out["e2e"] = {"value": e2e_value, "unit": "TFLOP/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "steps": n3, "call": "tiled_fp16_gemm_gb300.gemm_host",
                      "ms_per_step": dt / n3 * 1e3}
        del ha, hb
        bound = link_bound(h2d, d2h, device)
        bound["tflops_bound"] = flops / (bound["both_directions_ms"] / 1e3) / 1e12
        bound["frac"] = (e2e_value / world) / bound["tflops_bound"]
        out["e2e"]["bound"] = bound

    if _NVML is not None:
        _NVML.stop()

    # ---- CPU oracle on this host (rank 0, N == 1 only)
    if not args.no_cpu and rank == 0 and world == 1:
        tfl, rows, secs, th = cpu_oracle_rate(A, B, w, 12.0)
        out["cpu_baseline"] = {"value": tfl, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                               "sample": f"{rows} of {w.M} rows of {w.name} (full N, K), "
                                         f"{secs:.1f} s"}
    return out


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = rank_info()
    from tiled_fp16_gemm_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    from tiled_fp16_gemm_gb300 import build
    if rank == 0:
        build.build()
    if world > 1:
        barrier(world, None)
    out = run_ours(args, w, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
