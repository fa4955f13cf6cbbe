"""Throughput benchmark of tiled exact attention (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one forward pass plus one backward pass (all three backward
kernels) of the workload, on synthetic seeded bf16 inputs already resident in
HBM.  The L2 cache is flushed (256 MiB write) before every timed step; each
step is timed with CUDA events on the launching stream and the step time is
the sum of its event intervals.  Rank 0 prints one JSON line.

``--impl reference`` times the float64 CPU oracle on the host cores instead,
on a bounded sample of the same workload (one GQA group over a causal prefix),
in the same metric and unit.
"""
from __future__ import annotations

import argparse
import atexit
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

METRIC = "attention fwd+bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"

# DRAM bytes (read + write) of one launch of the dominant kernel, from one ncu
# capture of it on each workload listed.  Valid only for the kernel code it was
# taken on (comments aside): reported as null once that changes.
NCU_TRAFFIC = {
    "gqa_B2_H32x8_T8192_d128_causal": {"bytes": 729587200 + 349118720, "source_sha256_16": "1cbb8d11856b5dd4"},
    "swa_B1_H32x8_T8192_W2080_d128": {"bytes": 335243520 + 139563520, "source_sha256_16": "1cbb8d11856b5dd4"},
    "gqa_B1_H32x8_Tq4096_Tk8032_d128": {"bytes": 288794880 + 130316288, "source_sha256_16": "1cbb8d11856b5dd4"},
}
TRAFFIC_SOURCES = ("tiled_attention_05_gb300/csrc/fa_bwd.cu", "tiled_attention_05_gb300/csrc/sm103_ptx.cuh",
                   "tiled_attention_05_gb300/csrc/fa_internal.h")


def source_code_hash(paths=TRAFFIC_SOURCES) -> str:
    """sha256[:16] of the kernel sources with comments and whitespace removed,
    so that a comment-only edit does not detach a recorded measurement."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in paths:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    rec = NCU_TRAFFIC.get(workload)
    if rec is None:
        return None
    return rec["bytes"] if source_code_hash() == rec["source_sha256_16"] else None


FLUSH_BYTES = 256 << 20
# NVIDIA's nominal dense (no 2:4 sparsity) bf16 tensor peak of one GB300, in
# TFLOP/s.  The roofline uses the measured cuBLAS figure; the fraction of this
# nominal figure is reported beside it.
NOMINAL_BF16_DENSE_TFLOPS = 2250.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    return ap.parse_args(argv)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------- multi-rank plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, group_backend: str | None) -> float:
    """Max of a float over all ranks (identity for a single process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if group_backend == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, rank_seconds: float, world: int, backend: str | None) -> tuple:
    """Whole-job throughput: units processed by all ranks / max-over-ranks time."""
    t = reduce_max(rank_seconds, backend)
    return units_per_rank * world / t, t


# ---------------------------------------------------------------- clocks
class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver): the SM clock, its maximum, the power draw and the active
    clock-event (throttle) reasons of one GPU.  Nothing is ever set."""

    # nvmlClocksEventReason* bits (nvml.h)
    SW_POWER_CAP, HW_SLOWDOWN, SW_THERMAL, HW_THERMAL = 0x4, 0x8, 0x20, 0x40
    CLOCK_SM = 1

    def __init__(self, index: int):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.reasons_fn = fn
        self.max_mhz = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.CLOCK_SM)
        self.index = index

    def _uint(self, fn, *args):
        v = self.ct.c_uint()
        if fn(self.h, *args, self.ct.byref(v)) != 0:
            raise OSError("NVML query failed")
        return v.value

    def line(self) -> str:
        """One sample in the CSV form nvidia-smi prints for ClockSampler.FIELDS."""
        sm = self._uint(self.lib.nvmlDeviceGetClockInfo, self.CLOCK_SM)
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        r = self.ct.c_ulonglong()
        if self.reasons_fn(self.h, self.ct.byref(r)) != 0:
            raise OSError("NVML query failed")
        bits = r.value
        act = lambda b: "Active" if bits & b else "Not Active"  # noqa: E731
        return (f"{self.index}, {sm}, {self.max_mhz}, {mw / 1000.0:.2f}, 0x{bits:016x}, {act(self.HW_SLOWDOWN)}, "
                f"{act(self.HW_THERMAL)}, {act(self.SW_THERMAL)}, {act(self.SW_POWER_CAP)}")

    def close(self):
        try:
            self.lib.nvmlShutdown()
        except Exception:  # noqa: BLE001
            pass


class ClockSampler:
    """Samples the SM clock, power and throttle reasons of one GPU.

    It reads them through read-only NVML queries every 5 ms (falling back to
    nvidia-smi at 10 ms when NVML cannot be loaded), so that even a timed
    region of a few tens of milliseconds holds several samples.  It is started
    before the warm-up so that it is already sampling when the timed region
    begins; each sample is stamped with the host wall clock on arrival, and
    summary(t0, t1) keeps the samples taken inside [t0, t1].  A timed region
    shorter than the sampling period gets the two samples around it instead
    (both under load: warm-up before, end-to-end phase after), and the summary
    says so."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 5
    SMI_PERIOD_MS = 10

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.nvml = None
        self.stop = threading.Event()
        self.reader = None
        self.source = "none"
        self.lines = []  # (host time of arrival, csv line)

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.gpu_index)
            self.nvml.line()
            self.source = f"NVML every {self.PERIOD_MS} ms"
            self.reader = threading.Thread(target=self._poll, daemon=True)
            self.reader.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.SMI_PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = f"nvidia-smi every {self.SMI_PERIOD_MS} ms"
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def wait_live(self, timeout_s: float = 3.0):
        """Block until the first sample has arrived (or the timeout passes)."""
        t_end = time.time() + timeout_s
        while (self.proc is not None or self.nvml is not None) and not self.lines and time.time() < t_end:
            time.sleep(0.01)

    def _poll(self):
        while not self.stop.is_set():
            try:
                self.lines.append((time.time(), self.nvml.line()))
            except OSError:
                pass
            self.stop.wait(self.PERIOD_MS / 1000.0)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.reader is not None:
            self.reader.join(timeout=2)
        if self.nvml is not None:
            self.nvml.close()
            self.nvml = None

    def summary(self, t0: float | None = None, t1: float | None = None):
        window = "whole run"
        lines = self.lines
        if t0 is not None and t1 is not None:
            inside = [x for x in lines if t0 <= x[0] <= t1]
            if inside:
                lines, window = inside, "timed region"
            else:
                before = [x for x in lines if x[0] < t0][-1:]
                after = [x for x in lines if x[0] > t1][:1]
                lines = before + after
                window = f"the samples just before and after the timed region ({(t1 - t0) * 1e3:.0f} ms, " \
                         f"shorter than the sampling period)"
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0, "window": window}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "window": window, "source": self.source}


# ---------------------------------------------------------------- CPU oracle legs
def oracle_sample(w, rows: int | None, group: int = 0):
    """A bounded sample of the workload for the float64 oracle: one GQA group
    (batch group // Hkv, kv head group % Hkv, its G query heads) over all rows,
    or over the first `rows` tokens (a causal prefix, or the first `rows`
    queries against all keys).  Inputs are drawn with the workload's seed plus
    the group index."""
    from tiled_attention_05_gb300.inputs import Workload, make_custom

    G = w.G
    Tq = w.Tq if rows is None else min(rows, w.Tq)
    Tk = w.Tk if (rows is None or not w.causal) else min(rows, w.Tk)
    if w.causal and w.Tq != w.Tk and rows is not None:
        Tk = w.Tk - (w.Tq - Tq)
    Q, K, V, dO = make_custom(1, G, 1, Tq, Tk, w.d, w.causal, seed=w.seed + 1000 * group, dO_std=w.dO_std)
    sw = Workload("sample", 1, G, 1, Tq, Tk, w.d, w.causal, w.seed, window=w.window)
    return (Q, K, V, dO), sw


def time_oracle(w, rows, nthreads, group: int = 0):
    import oracle

    (Q, K, V, dO), sw = oracle_sample(w, rows, group)
    Qn, Kn, Vn, dOn = (oracle._f64(t) for t in (Q, K, V, dO))
    t0 = time.perf_counter()
    oracle.forward(Qn, Kn, Vn, w.causal, nthreads=nthreads, window=w.window)
    oracle.backward(Qn, Kn, Vn, dOn, w.causal, nthreads=nthreads, window=w.window)
    dt = time.perf_counter() - t0
    return sw.flops("fwdbwd"), dt, sw


def cpu_baseline_leg(w, cores, min_seconds=10.0):
    """Oracle fwd+bwd over whole GQA groups of the workload until `min_seconds`
    of CPU work (or every group) is done."""
    flops, secs, n = 0.0, 0.0, 0
    groups = w.B * w.Hkv
    while n < groups and secs < min_seconds:
        f, dt, sw = time_oracle(w, None, cores, group=n)
        flops, secs, n = flops + f, secs + dt, n + 1
    # context: the same oracle on one core, over a 2048-token prefix of one group
    f1, dt1, sw1 = time_oracle(w, 2048, 1)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {groups} GQA groups ({w.G} query heads each, all {w.Tq} rows, Tk={w.Tk}); "
                      f"float64 forward + backward; {secs:.1f} s",
            "one_core": {"value": f1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                         "sample": f"one GQA group, Tq={sw1.Tq}, Tk={sw1.Tk}; {dt1:.1f} s"}}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm
def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cores = host_cores()
    rows = 2048 if w.Tq > 2048 else None
    flops_sum, secs = 0.0, 0.0
    sw = None
    for i in range(args.warmup + args.steps):
        f, dt, sw = time_oracle(w, rows, cores)
        if i >= args.warmup:
            flops_sum += f
            secs += dt
    value = flops_sum / secs / 1e12
    sample = (f"one GQA group (batch 0, kv head 0, {w.G} query heads), Tq={sw.Tq}, Tk={sw.Tk}, d={w.d}, "
              f"causal={w.causal}, window={w.window}; float64 forward + backward")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Tq": w.Tq, "Tk": w.Tk, "d": w.d,
                       "causal": w.causal, "window": w.window},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import tiled_attention_05_gb300 as fa
    from tiled_attention_05_gb300.inputs import make_inputs

    world, rank, local = dist_env()
    backend = None
    if world > 1:
        backend = "nccl"
        torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()
    peaks = load_peaks()

    Qh, Kh, Vh, dOh = make_inputs(w)
    Q, K, V, dO = (t.to(dev) for t in (Qh, Kh, Vh, dOh))
    O = torch.empty_like(dO)  # [B, Hq, Tq, dv]
    L = torch.empty(w.B, w.Hq, w.Tq, dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dims = fa.make_dims(w.B, w.Hq, w.Hkv, w.Tq, w.Tk, w.d, w.dv, w.causal, None, w.window)
    ws = torch.empty(fa.fa_backward_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        launches = 0
        if evs:
            evs[0].record(stream)
        fa.fa_forward(Q, K, V, w.causal, None, O=O, L=L, window=w.window)
        launches += fa.last_launch_count()
        if evs:
            evs[1].record(stream)
        fa.fa_backward(Q, K, V, O, dO, L, w.causal, None, dQ, dK, dV, ws, stages=fa.FA_BWD_PRE, window=w.window)
        launches += fa.last_launch_count()
        if evs:
            evs[2].record(stream)
        fa.fa_backward(Q, K, V, O, dO, L, w.causal, None, dQ, dK, dV, ws, stages=fa.FA_BWD_MAIN, window=w.window)
        launches += fa.last_launch_count()
        if evs:
            evs[3].record(stream)
        fa.fa_backward(Q, K, V, O, dO, L, w.causal, None, dQ, dK, dV, ws, stages=fa.FA_BWD_CAST, window=w.window)
        launches += fa.last_launch_count()
        if evs:
            evs[4].record(stream)
        return launches

    clocks = ClockSampler(local)  # sampling from the warm-up through the end-to-end phase
    clocks.__enter__()
    atexit.register(clocks.__exit__, None, None, None)  # also on an error exit
    clocks.wait_live()
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("kernel timeout during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    launches = 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_region0 = time.time()
    t_wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        launches += step(evs[k])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    t_region1 = time.time()
    if world > 1:
        dist.barrier()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("kernel timeout in the timed region")

    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    pre_ms = [e[1].elapsed_time(e[2]) for e in evs]
    main_ms = [e[2].elapsed_time(e[3]) for e in evs]
    cast_ms = [e[3].elapsed_time(e[4]) for e in evs]
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    rank_secs = sum(step_ms) / 1e3
    flops_step = w.flops("fwdbwd")
    value_flops, t_max = aggregate_throughput(flops_step * args.steps, rank_secs, world, backend)
    value = value_flops / 1e12
    bwd_ms = [a + b + c for a, b, c in zip(pre_ms, main_ms, cast_ms)]
    fwd_tflops = w.flops("fwd") / (statistics.mean(fwd_ms) / 1e3) / 1e12
    bwd_tflops = w.flops("bwd") / (statistics.mean(bwd_ms) / 1e3) / 1e12
    main_tflops = w.flops("bwd") / (statistics.mean(main_ms) / 1e3) / 1e12

    # ---- end to end through the public API with host buffers (pinned), same metric.
    # Every step uploads its inputs (Q, K, V, dO) from pinned host memory and
    # reads its results (dQ, dK, dV) back.  Uploads and read-backs run on
    # their own streams into double-buffered device tensors, so step k's
    # compute overlaps step k+1's upload and step k-1's read-back.
    pin = [t.pin_memory() for t in (Qh, Kh, Vh, dOh)]
    outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (Qh, Kh, Vh)]
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = []
    for i in range(2):
        if i == 0:
            ins, res = [Q, K, V, dO], [dQ, dK, dV]
        else:
            ins, res = [torch.empty_like(t) for t in (Q, K, V, dO)], [torch.empty_like(t) for t in (dQ, dK, dV)]
        sets.append({"in": ins, "res": res, "O": torch.empty_like(O), "L": torch.empty_like(L),
                     "ws": ws if i == 0 else torch.empty_like(ws),
                     "uploaded": torch.cuda.Event(), "computed": torch.cuda.Event(), "read": torch.cuda.Event()})

    def e2e_steps(n):
        for k in range(n):
            st_ = sets[k % 2]
            with torch.cuda.stream(s_up):
                if k >= 2:
                    s_up.wait_event(st_["computed"])  # step k-2 no longer reads these inputs
                for dst, src in zip(st_["in"], pin):
                    dst.copy_(src, non_blocking=True)
                st_["uploaded"].record(s_up)
            stream.wait_event(st_["uploaded"])
            if k >= 2:
                stream.wait_event(st_["read"])  # step k-2's results have been read back
            q, kk, v, g = st_["in"]
            fa.fa_forward(q, kk, v, w.causal, None, O=st_["O"], L=st_["L"], stream=stream, window=w.window)
            fa.fa_backward(q, kk, v, st_["O"], g, st_["L"], w.causal, None, *st_["res"], st_["ws"], stream=stream,
                           window=w.window)
            st_["computed"].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(st_["computed"])
                for dst, src in zip(outs, st_["res"]):
                    dst.copy_(src, non_blocking=True)
                st_["read"].record(s_down)

    e2e_steps(max(2, args.warmup))
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e_start.record(stream)
    s_up.wait_event(e_start)
    e2e_steps(args.steps)
    s_down.wait_event(sets[(args.steps - 1) % 2]["read"])
    e_end.record(s_down)
    torch.cuda.synchronize()
    e2e_secs = e_start.elapsed_time(e_end) / 1e3
    clocks.__exit__(None, None, None)
    e2e_value, _ = aggregate_throughput(flops_step * args.steps, e2e_secs, world, backend)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(w, host_cores())

    peak = peaks["bf16_tflops"]
    frac = main_tflops / peak
    if rank == 0:
        clk = clocks.summary(t_region0, t_region1)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Tq": w.Tq, "Tk": w.Tk, "d": w.d,
                       "causal": w.causal, "window": w.window, "parallelism": "replicas" if world > 1 else "single",
                       "l2": "flushed before every timed step (256 MiB write)"},
            "pct_of_peak": 100.0 * value / peak,
            "pct_of_nominal_peak": 100.0 * value / NOMINAL_BF16_DENSE_TFLOPS,
            "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
            "fwd_ms": statistics.mean(fwd_ms), "bwd_ms": statistics.mean(bwd_ms),
            "bwd_stage_ms": {"pre": statistics.mean(pre_ms), "main": statistics.mean(main_ms),
                             "cast": statistics.mean(cast_ms)},
            "roofline": {"kernel": "fa_bwd_main", "bound": "tensor", "achieved": main_tflops, "peak": peak,
                         "unit": "TFLOP/s", "frac": frac, "traffic": measured_traffic(w.name),
                         "peak_source": f"{peaks['source']} bf16 burst"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_secs / args.steps * 1e3,
                    "copies": "pinned host <-> device on two copy streams, overlapped with compute"},
            "gpu_launches": launches,
            "clocks": clk,
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    from tiled_attention_05_gb300.inputs import HEADLINE, WORKLOADS

    w = WORKLOADS[args.workload or HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
