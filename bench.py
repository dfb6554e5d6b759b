"""Throughput of the dense GEMM C = A * B^T (and the decode GEMV) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra] [--no-cpu-baseline]

One step is one C = A * B^T over the workload's seeded synthetic operands,
already resident in HBM: one launch of the planned kernel.  The default
workload is the 8192^3 bf16 -> bf16 GEMM.  Prints ONE JSON line (rank 0).

--impl reference times the CPU oracle (plain fp64 triple loop, OpenMP over
rows) on a bounded row sample of the same workload, in the same metric.

Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU (the output tiles are independent; there is no data exchange), the
timed region is bracketed by a barrier and device synchronisation, the
maximum elapsed time over ranks is taken, and the value counts the work of
all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from dense_gemm_blackwell_sm_gb300 import inputs, roofline  # noqa: E402

METRIC = "GEMM TFLOP/s (and % of dense peak) at 4096³/8192³ bf16; GEMV GB/s"
DEFAULT_WORKLOAD = "large_8192_bf16_bf16"
STATED_PEAK_TFLOPS = 2000.0   # the pages' B200 FP16 figure, used as the stated target
STATED_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# source files whose change invalidates a stored ncu traffic figure
KERNEL_SOURCES = {
    "ws": ["dense_gemm_blackwell_sm_gb300/csrc/kernels_ws.cu", "dense_gemm_blackwell_sm_gb300/csrc/kernels_ws.cuh",
           "dense_gemm_blackwell_sm_gb300/csrc/ptx.cuh", "dense_gemm_blackwell_sm_gb300/csrc/kernel_common.cuh"],
    "mx": ["dense_gemm_blackwell_sm_gb300/csrc/kernels_mx.cu", "dense_gemm_blackwell_sm_gb300/csrc/kernels_ws.cuh",
           "dense_gemm_blackwell_sm_gb300/csrc/ptx.cuh", "dense_gemm_blackwell_sm_gb300/csrc/kernel_common.cuh"],
    "gemv": ["dense_gemm_blackwell_sm_gb300/csrc/kernel_gemv.cu", "dense_gemm_blackwell_sm_gb300/csrc/kernel_gemv_tc.cu",
             "dense_gemm_blackwell_sm_gb300/csrc/kernel_common.cuh", "dense_gemm_blackwell_sm_gb300/csrc/ptx.cuh"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


# ---------------------------------------------------------------------------
# host helpers (importable without a GPU)

def measured_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK), "fallback"


def code_tokens(src: str) -> str:
    """A C++/CUDA source without its comments and with runs of whitespace collapsed:
    what decides whether a kernel changed (string literals hold no comment markers in
    these files)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def source_hash(kind: str) -> str:
    """First 16 hex digits of the sha256 of the kernel sources' code (comments and
    layout left out), recorded with each ncu traffic capture."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel is unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(kind, {}).get(workload)
        if e and e.get("source_hash") == source_hash(kind):
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def aggregate(per_rank_seconds: list[float], units_per_rank: float) -> tuple[float, float]:
    """(max elapsed over ranks, whole-job units per second)."""
    t = max(per_rank_seconds)
    return t, units_per_rank * len(per_rank_seconds) / t


class ClockSampler:
    """nvidia-smi clocks / power / throttle reasons sampled every 50 ms while
    work runs.  Each sample carries nvidia-smi's own timestamp, so a summary
    can be restricted to the host-time window of one timed region.  power.draw
    is averaged over about a second, so a timed region of a tenth of a second
    barely moves it; where the driver offers power.draw.instant, that decides
    whether a sample was under load."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,enforced.power.limit,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def _start(self, query: str) -> bool:
        """Start nvidia-smi on `query`; True once it produces samples."""
        self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + query,
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        # NVML start-up can hold the driver for a moment: start timing only
        # once the sampler is producing samples
        t0 = time.time()
        while not self.lines and time.time() - t0 < 10.0 and self.proc.poll() is None:
            time.sleep(0.02)
        ok = bool(self.parse(self.lines[:1]))
        if not ok:
            self._stop()
            self.lines = []
        return ok

    def __enter__(self):
        try:
            if not self._start(self.QUERY + ",power.draw.instant"):
                self._start(self.QUERY)
            time.sleep(0.1)
        except OSError:
            self.proc = None
        return self

    def _stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self._stop()
        return False

    @staticmethod
    def parse(lines: list[str]) -> list[dict]:
        out = []
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 11:
                continue
            try:
                t = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                if "." in f[0]:
                    t += float("0." + f[0].split(".")[1])
                smp = {"t": t, "mhz": float(f[2]), "max_mhz": float(f[3])}
            except ValueError:
                continue
            try:
                smp["w"] = float(f[4])
                smp["limit_w"] = float(f[5])
            except ValueError:
                smp["w"], smp["limit_w"] = None, None
            smp["w_inst"] = None
            if len(f) > 11:
                try:
                    smp["w_inst"] = float(f[11])
                except ValueError:
                    pass
            smp["reasons"] = [n for n, v in zip(ClockSampler.REASONS, f[7:11]) if v.lower().startswith("active")]
            out.append(smp)
        return out

    def summary(self, t0: float | None = None, t1: float | None = None) -> dict:
        """Median SM clock (all samples and those under load), power and throttle
        reasons, over the samples within [t0, t1] (host time.time()) if given.
        A sample is under load when it draws more than 40 % of the power limit
        (instantaneous power where sampled, else the averaged draw)."""
        smp = self.parse(self.lines)
        if t0 is not None:
            smp = [x for x in smp if t0 - 0.05 <= x["t"] <= t1 + 0.05]
        if not smp:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        mhz = sorted(x["mhz"] for x in smp)

        def watts(x):
            return x["w_inst"] if x.get("w_inst") is not None else x["w"]

        load = sorted(x["mhz"] for x in smp if watts(x) is not None and x["limit_w"] and watts(x) > 0.4 * x["limit_w"])
        reasons = sorted({r for x in smp for r in x["reasons"]})
        pw = [x["w"] for x in smp if x["w"] is not None]
        pi = [x["w_inst"] for x in smp if x.get("w_inst") is not None]
        out = {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(x["max_mhz"] for x in smp), "reasons": reasons,
               "samples": len(smp), "samples_under_load": len(load),
               "sm_mhz_under_load": load[len(load) // 2] if load else None,
               "power_w_max": max(pw) if pw else None, "power_limit_w": smp[-1]["limit_w"]}
        if pi:
            out["power_w_instant_max"] = max(pi)
        return out


# ---------------------------------------------------------------------------
# GPU timing

def _events_time(fn, steps: int, stream) -> float:
    """Seconds for `steps` calls of fn(i) on `stream`, CUDA events on that stream."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def bench_gemm(w: inputs.Workload, steps: int, warmup: int, dev, dist_barrier, variant: int = 0,
               epilogue_act=None) -> dict:
    """Average launch time of the planned GEMM.  With ``epilogue_act`` set, the
    fused epilogue act(A B^T + bias) + residual runs in the same launch."""
    from dense_gemm_blackwell_sm_gb300 import gemm
    code = gemm.dtype_code(w.in_dtype, w.out_dtype)
    a, b = inputs.workload_operands(w)
    mx = w.in_dtype in (inputs.MXE4M3, inputs.MXE5M2)
    if mx:   # block scales in the kernels' tiled layout, resident like the operands
        sfa, sfb = inputs.workload_mx_scales(w)
        sfa, sfb = inputs.mx_tile_scales(sfa, w.K).to(dev), inputs.mx_tile_scales(sfb, w.K).to(dev)
    # operand sets used in turn, together larger than twice the L2 (two for the large
    # workloads, whose inputs alone exceed it), so no launch finds its inputs in L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = a.numel() * a.element_size() + b.numel() * b.element_size()
    nsets = max(2, int((2 * l2 + set_bytes - 1) // set_bytes))
    sets = []
    for s in range(nsets):
        sets.append((a.to(dev), b.to(dev), torch.empty((w.M, w.N), device=dev, dtype=inputs.torch_dtype(w.out_dtype))))
    plan = gemm.Plan(w.M, w.N, w.K, code, gemm.make_opts(variant=variant))
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ptrs = [(x.data_ptr(), y.data_ptr(), z.data_ptr()) for x, y, z in sets]
    epi = None
    lib = gemm.load()
    import ctypes
    if epilogue_act is not None:
        bias = torch.randn(w.N, device=dev, dtype=torch.float32)
        res = torch.randn(w.M, w.N, device=dev).to(inputs.torch_dtype(w.out_dtype))
        epi = gemm.Epilogue()
        epi.bias, epi.residual, epi.activation = bias.data_ptr(), res.data_ptr(), int(epilogue_act)

    def step(i):
        pa, pb, pc = ptrs[i % nsets]
        if mx:
            st = lib.gemm_plan_run_mx(plan._h, pa, pb, pc, sfa.data_ptr(), sfb.data_ptr(),
                                      None if epi is None else ctypes.byref(epi), sp)
        elif epi is None:
            st = plan.run_ptr(pa, pb, pc, sp)
        else:
            st = lib.gemm_plan_run_epilogue(plan._h, pa, pb, pc, ctypes.byref(epi), sp)
        if st != 0:
            raise gemm.GemmError(st, "gemm_plan_run")

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    assert plan.check() == gemm.OK
    dist_barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        h0 = time.time()
        secs = _events_time(step, steps, stream)
        h1 = time.time()
    torch.cuda.synchronize(dev)
    dist_barrier()
    st = plan.check()
    if st != gemm.OK:
        raise gemm.GemmError(st, "device status after the timed region")
    info = plan.info()
    plan.destroy()
    del sets
    clocks = clk.summary(h0, h1)
    clocks["scope"] = "timed region"
    if clocks["samples"] == 0:
        # the region is shorter than one 50 ms sample: report the sampler's whole run
        clocks = clk.summary()
        clocks["scope"] = "sampler run around a timed region shorter than one sample"
    return {"seconds": secs, "per_launch_s": secs / steps, "clocks": clocks, "info": info,
            "operand_sets": nsets}


def bench_gemm_e2e(w: inputs.Workload, steps: int, dev) -> dict:
    """The same GEMM through gemm_run_host: pinned host operands in, host result out.
    Block-scaled workloads (no host entry point) copy operands and scales in with
    torch from pinned memory, run gemm_plan_run_mx and copy C back, every step."""
    from dense_gemm_blackwell_sm_gb300 import gemm
    code = gemm.dtype_code(w.in_dtype, w.out_dtype)
    a, b = inputs.workload_operands(w)
    ib = 1 if w.in_dtype in inputs.EIGHT_BIT else 2
    ob = 4 if w.out_dtype == "f32" else 2
    if w.in_dtype in (inputs.MXE4M3, inputs.MXE5M2):
        return _bench_mx_e2e(w, a, b, code, steps, dev, ib, ob)
    ah, bh = a.pin_memory(), b.pin_memory()
    ch = torch.empty((w.M, w.N), dtype=inputs.torch_dtype(w.out_dtype)).pin_memory()
    da, db = torch.empty_like(a, device=dev), torch.empty_like(b, device=dev)
    dc = torch.empty((w.M, w.N), device=dev, dtype=inputs.torch_dtype(w.out_dtype))
    sp = torch.cuda.current_stream(dev).cuda_stream

    def once():
        st = gemm.gemm_run_host(w.M, w.N, w.K, ah.data_ptr(), bh.data_ptr(), ch.data_ptr(), code,
                                da.data_ptr(), db.data_ptr(), dc.data_ptr(), sp)
        if st != 0:
            raise gemm.GemmError(st, "gemm_run_host")

    once()
    # three timed windows of `steps` steps; the median window is reported (one window
    # alone has shown a host hiccup of ~10 ms inflating a 1.6 ms step by 65 %)
    windows = []
    for _ in range(3):
        t0 = time.perf_counter()
        for _ in range(steps):
            once()   # synchronises the stream itself
        windows.append(time.perf_counter() - t0)
    secs = sorted(windows)[1]
    return {"seconds": secs, "steps": steps, "h2d": ib * (w.M * w.K + w.N * w.K), "d2h": ob * w.M * w.N,
            "window_ms_per_step": [round(x / steps * 1e3, 3) for x in windows],
            "copy_only": copy_ceiling(dev, [(ah, da), (bh, db)], [(ch, dc)])}


def copy_ceiling(dev, h2d: list, d2h: list, reps: int = 5) -> dict:
    """The host-link floor of one end-to-end step: the same bytes copied in
    (pinned host -> device) and out (device -> pinned host) on two streams at
    once, with no GEMM; best of `reps`.  Also each direction alone."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(do_in, do_out):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if do_in:
                with torch.cuda.stream(s_in):
                    for h, d in h2d:
                        d.copy_(h, non_blocking=True)
            if do_out:
                with torch.cuda.stream(s_out):
                    for h, d in d2h:
                        h.copy_(d, non_blocking=True)
            torch.cuda.synchronize(dev)
            t = time.perf_counter() - t0
            best = t if best is None else min(best, t)
        return best
    bi = sum(h.numel() * h.element_size() for h, _ in h2d)
    bo = sum(h.numel() * h.element_size() for h, _ in d2h)
    t_in, t_out, t_both = run(True, False), run(False, True), run(True, True)
    return {"ms_both": round(t_both * 1e3, 3), "ms_in": round(t_in * 1e3, 3), "ms_out": round(t_out * 1e3, 3),
            "gbs_in": round(bi / t_in / 1e9, 1), "gbs_out": round(bo / t_out / 1e9, 1)}


def _bench_mx_e2e(w, a, b, code, steps, dev, ib, ob) -> dict:
    from dense_gemm_blackwell_sm_gb300 import gemm
    sfa, sfb = inputs.workload_mx_scales(w)
    host = [x.pin_memory() for x in (a, b, inputs.mx_tile_scales(sfa, w.K), inputs.mx_tile_scales(sfb, w.K))]
    devs = [torch.empty_like(x, device=dev) for x in host]
    ch = torch.empty((w.M, w.N), dtype=inputs.torch_dtype(w.out_dtype)).pin_memory()
    dc = torch.empty((w.M, w.N), device=dev, dtype=inputs.torch_dtype(w.out_dtype))
    plan = gemm.Plan(w.M, w.N, w.K, code)

    def once():
        for d, h in zip(devs, host):
            d.copy_(h, non_blocking=True)
        plan.run_mx(devs[0], devs[1], dc, devs[2], devs[3])
        ch.copy_(dc, non_blocking=True)
        torch.cuda.synchronize(dev)

    once()
    windows = []  # as in bench_gemm_e2e: the median of three timed windows
    for _ in range(3):
        t0 = time.perf_counter()
        for _ in range(steps):
            once()
        windows.append(time.perf_counter() - t0)
    secs = sorted(windows)[1]
    plan.destroy()
    return {"seconds": secs, "steps": steps, "h2d": sum(x.numel() * x.element_size() for x in host),
            "d2h": ob * w.M * w.N, "window_ms_per_step": [round(x / steps * 1e3, 3) for x in windows]}


def bench_gemv(w: inputs.Workload, steps: int, warmup: int, dev, flags: int = 0, variant: int = 0) -> dict:
    """GB/s of the decode GEMV (automatic plan unless `variant` is given).  The weight rotates over enough
    copies to exceed 4x L2, and the launches are captured in a CUDA graph so that
    the host's launch cost does not stand between these few-microsecond kernels."""
    from dense_gemm_blackwell_sm_gb300 import gemm
    code = gemm.dtype_code(w.in_dtype, w.out_dtype)
    x, b = inputs.workload_operands(w)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    wbytes = b.numel() * 2
    copies = max(2, int((4 * l2 + wbytes - 1) // wbytes))
    xs = x.to(dev)
    bs = [b.to(dev) for _ in range(copies)]
    ys = [torch.empty((w.M, w.N), device=dev, dtype=inputs.torch_dtype(w.out_dtype)) for _ in range(copies)]
    plan = gemm.Plan(w.M, w.N, w.K, code, gemm.make_opts(flags=flags, variant=variant))
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    ptrs = [(xs.data_ptr(), bb.data_ptr(), yy.data_ptr()) for bb, yy in zip(bs, ys)]
    with torch.cuda.stream(stream):
        for i in range(warmup):
            assert plan.run_ptr(*ptrs[i % copies], sp) == 0
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            assert plan.run_ptr(*ptrs[i % copies], stream.cuda_stream) == 0
    with torch.cuda.stream(stream):
        graph.replay()
        secs = _events_time(lambda i: graph.replay(), 3, stream)
    assert plan.check(stream=stream) == gemm.OK
    info = plan.info()
    plan.destroy()
    del graph
    nbytes = roofline.gemm_bytes(w.M, w.N, w.K, 2, 4 if w.out_dtype == "f32" else 2)
    per = secs / (3 * steps)
    return {"gbs": nbytes / per / 1e9, "us_per_launch": per * 1e6, "copies": copies,
            "bytes_per_launch": nbytes, "variant": info["variant_name"]}


# ---------------------------------------------------------------------------
# CPU oracle timing (a reported baseline, not the target)

def host_cpu() -> dict:
    """The host CPU: model name (lscpu, else /proc/cpuinfo), the cores this
    process may run on (affinity) and the logical CPU count."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    try:
        aff = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        aff = os.cpu_count() or 0
    return {"model": model or platform.processor() or "unknown", "machine": platform.machine(),
            "affinity_cores": aff, "logical_cpus": os.cpu_count() or 0}


def oracle_steps(w: inputs.Workload, steps: int, warmup: int, step_s: float) -> dict:
    """The CPU oracle as a sequence of steps, each a bounded sample of the
    workload: the same number of seeded random rows of C (all N columns) per
    step, chosen from the first warm-up step so that one step takes about
    `step_s` seconds on all host threads.  Returns the timed steps' totals."""
    import numpy as np
    import oracle
    oracle.build()
    a, b = inputs.workload_operands(w)
    mx = w.in_dtype in (inputs.MXE4M3, inputs.MXE5M2)
    if mx:
        sfa, sfb = inputs.workload_mx_scales(w)
    threads = oracle.max_threads()
    rng = np.random.default_rng(0)

    def step(nrows):
        rows = rng.choice(w.M, size=min(nrows, w.M), replace=False)
        t0 = time.perf_counter()
        if mx:
            oracle.gemm_mx(a, b, sfa, sfb, rows=rows, nthreads=threads)
        else:
            oracle.gemm_rows(a, b, rows, nthreads=threads)
        return time.perf_counter() - t0, len(rows)

    t_cal, n_cal = step(threads)   # first warm-up step: one row per thread
    rows = max(1, min(w.M, int(n_cal * step_s / max(t_cal, 1e-6))))
    for _ in range(max(0, warmup - 1)):
        step(rows)
    t_tot, r_tot = 0.0, 0
    for _ in range(steps):
        t, n = step(rows)
        t_tot += t
        r_tot += n
    return {"tflops": 2.0 * r_tot * w.N * w.K / t_tot / 1e12, "seconds": t_tot, "rows_per_step": rows,
            "threads": threads}


def cpu_oracle_rate(w: inputs.Workload, budget_s: float = 12.0) -> dict:
    import numpy as np
    import oracle
    oracle.build()
    a, b = inputs.workload_operands(w)
    mx = w.in_dtype in (inputs.MXE4M3, inputs.MXE5M2)
    if mx:
        sfa, sfb = inputs.workload_mx_scales(w)
    threads = oracle.max_threads()
    rng = np.random.default_rng(0)
    rows_done, t_spent, batch = 0, 0.0, max(1, threads)
    while t_spent < budget_s and rows_done < w.M:
        rows = rng.choice(w.M, size=min(batch, w.M - rows_done), replace=False)
        t0 = time.perf_counter()
        if mx:
            oracle.gemm_mx(a, b, sfa, sfb, rows=rows, nthreads=threads)
        else:
            oracle.gemm_rows(a, b, rows, nthreads=threads)
        t_spent += time.perf_counter() - t0
        rows_done += len(rows)
        if t_spent < budget_s / 4:
            batch *= 2
    flops = 2.0 * rows_done * w.N * w.K
    # the same oracle on one thread, over a short fixed sample (a few seconds)
    t1, rows1 = 0.0, 0
    while t1 < budget_s / 6 and rows1 < w.M:
        r1 = [int(rng.integers(0, w.M))]
        t0 = time.perf_counter()
        if mx:
            oracle.gemm_mx(a, b, sfa, sfb, rows=r1, nthreads=1)
        else:
            oracle.gemm_rows(a, b, r1, nthreads=1)
        t1 += time.perf_counter() - t0
        rows1 += 1
    return {"tflops": flops / t_spent / 1e12, "rows": rows_done, "seconds": t_spent, "threads": threads,
            "single_thread_tflops": 2.0 * rows1 * w.N * w.K / t1 / 1e12, "single_thread_rows": rows1,
            "host": host_cpu(),
            "sample": "%d of %d rows of C (all %d columns, K=%d), seeded random rows, fp64 oracle on %d host "
                      "threads; rate extrapolates linearly to the full %dx%dx%d product" % (
                          rows_done, w.M, w.N, w.K, threads, w.M, w.N, w.K)}


# ---------------------------------------------------------------------------

def _g_act_silu() -> int:
    from dense_gemm_blackwell_sm_gb300 import gemm
    return gemm.ACT_SILU


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0, (lambda: None), (lambda x: [x])
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend)

    def barrier():
        dist.barrier()

    def gather(x: float):
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if backend == "nccl" else "cpu")
        out = [torch.zeros_like(t) for _ in range(ws)]
        dist.all_gather(out, t)
        return [float(o.item()) for o in out]
    return rank, ws, local, barrier, gather


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--epilogue", default=None, choices=["none", "relu", "silu", "gelu_tanh", "gelu_erf"],
                    help="time the step with the fused epilogue act(A B^T + bias) + residual")
    ap.add_argument("--shape", default=None,
                    help="M,N,K[,in,out]: a custom bf16 GEMM shape instead of a named workload (profiling)")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--ladder", action="store_true",
                    help="time every kernel variant (the nine steps) on the workload and print one JSON line per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    w = inputs.WORKLOADS[args.workload]
    if args.shape:
        f = args.shape.split(",")
        M, N, K = (int(x) for x in f[:3])
        ti, to = (f[3], f[4]) if len(f) >= 5 else ("bf16", "bf16")
        w = inputs.Workload("custom_%dx%dx%d_%s_%s" % (M, N, K, ti, to), M, N, K, ti, to,
                            inputs.N002, inputs.N002, 7)
    rank, world, local, barrier, gather = _dist()

    if args.impl == "reference":
        if rank != 0:
            return 0
        # every step is the same bounded row sample; all steps together take about a minute
        step_s = min(3.0, 60.0 / max(1, args.steps + args.warmup))
        r = oracle_steps(w, args.steps, args.warmup, step_s)
        host = host_cpu()
        sample = ("each step: %d seeded random rows of C (all %d columns, K=%d) of the %dx%dx%d product, "
                  "fp64 oracle on %d host threads" % (r["rows_per_step"], w.N, w.K, w.M, w.N, w.K, r["threads"]))
        line = {"impl": "reference", "metric": METRIC, "value": round(r["tflops"], 6), "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(r["seconds"] / args.steps * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in": w.in_dtype, "out": w.out_dtype,
                           "rows_per_step": r["rows_per_step"]},
                "cpu_baseline": {"value": round(r["tflops"], 6), "unit": "TFLOP/s", "cores": r["threads"],
                                 "host": host, "kind": "oracle", "sample": sample},
                "e2e": {"value": round(r["tflops"], 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()

    if args.ladder:
        from dense_gemm_blackwell_sm_gb300 import gemm as _g
        for v in range(_g.S3, _g.S9 + 1):
            r = bench_gemm(w, args.steps, args.warmup, dev, lambda: None, v)
            print(json.dumps({"ladder_step": v, "variant": r["info"]["variant_name"], "workload": w.name,
                              "tflops": round(w.flops / r["per_launch_s"] / 1e12, 1),
                              "us_per_launch": round(r["per_launch_s"] * 1e6, 1), "grid": r["info"]["grid"],
                              "stages": r["info"]["stages"], "clocks": r["clocks"]}), flush=True)
        return 0

    epi_act = None
    if args.epilogue is not None:
        epi_act = ["none", "relu", "silu", "gelu_tanh", "gelu_erf"].index(args.epilogue)
    res = bench_gemm(w, args.steps, args.warmup, dev, barrier, args.variant, epilogue_act=epi_act)
    times = gather(res["seconds"])
    tmax, flops_per_s = aggregate(times, w.flops * args.steps)
    tflops = flops_per_s / 1e12
    per_launch = res["per_launch_s"]

    peaks, peak_src = measured_peaks()
    long_region = res["seconds"] > 2.0
    peak_key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    # fp16 and bf16 run at the same dense Tensor Core rate; 8-bit floats at twice it
    # (the nominal fp8 / bf16 dense ratio, 4.5 / 2.25 PFLOP/s, times the measured bf16 peak)
    peak = float(peaks.get(peak_key, FALLBACK[peak_key]))
    if w.in_dtype in inputs.EIGHT_BIT:
        peak *= 2.0
        peak_key += " x 2 (fp8)"
    achieved = w.flops / per_launch / 1e12
    stated = STATED_PEAK_TFLOPS * (2 if w.in_dtype in inputs.EIGHT_BIT else 1)
    line = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tmax / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.in_dtype, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in": w.in_dtype, "out": w.out_dtype,
                   "variant": res["info"]["variant_name"], "tile": [res["info"]["tile_m"], res["info"]["tile_n"]],
                   "cluster": res["info"]["cluster"], "stages": res["info"]["stages"],
                   "grid": res["info"]["grid"], "sched": res["info"]["sched"],
                   "epilogue": args.epilogue or "plain",
                   "l2": "inputs larger than L2: %d operand sets of A+B+C = %d MB used in turn" % (
                       res["operand_sets"], w.algorithmic_bytes // 2**20),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": stored_traffic("mx" if w.in_dtype in (inputs.MXE4M3, inputs.MXE5M2) else "ws", w.name),
                     "peak_source": "%s %s" % (peak_key, peak_src),
                     "frac_of_stated_%d" % stated: round(achieved / stated, 4)},
        "clocks": res["clocks"],
        "gpu_launches": args.steps,
    }
    if rank == 0 and not args.no_e2e:
        e = bench_gemm_e2e(w, max(3, min(10, args.steps // 20)), dev)
        line["e2e"] = {"value": round(w.flops * e["steps"] / e["seconds"] / 1e12, 3), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": round(e["seconds"] / e["steps"] * 1e3, 3)}
        if e.get("window_ms_per_step"):
            line["e2e"]["timing"] = "median of 3 windows of %d steps" % e["steps"]
            line["e2e"]["window_ms_per_step"] = e["window_ms_per_step"]
        if e.get("copy_only"):
            c = e["copy_only"]
            # the step can finish no sooner than its copies alone (both directions at once)
            line["e2e"]["copy_only_ceiling"] = dict(c, tflops=round(w.flops / (c["ms_both"] * 1e-3) / 1e12, 3),
                                                    frac=round(c["ms_both"] / line["e2e"]["ms_per_step"], 4))
    if rank == 0 and not args.no_extra:
        also = {}
        # the same step back to back for at least 3 s, against the sustained peak,
        # with the clocks and power seen under load
        n_sus = max(args.steps, int(3.2 / max(per_launch, 1e-6)))
        rs = bench_gemm(w, n_sus, 10, dev, lambda: None, args.variant, epilogue_act=epi_act)
        ts = w.flops / rs["per_launch_s"] / 1e12
        sus_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"]))
        if w.in_dtype in inputs.EIGHT_BIT:
            sus_peak *= 2.0
        ck = rs["clocks"]
        also["sustained_" + w.name] = {
            "tflops": round(ts, 3), "launches": n_sus, "seconds": round(rs["seconds"], 3),
            "peak": sus_peak, "peak_source": "bf16_tflops_sustained %s" % peak_src, "frac": round(ts / sus_peak, 4),
            "clocks": ck,
            # time x clock: launch time normalised to the median SM clock under load
            "us_x_ghz": round(rs["per_launch_s"] * 1e6 * (ck.get("sm_mhz_under_load") or ck.get("sm_mhz") or 0) / 1e3, 1)}
        w3 = inputs.WORKLOADS["square_4096_f16_f32"]
        r3 = bench_gemm(w3, 200, 10, dev, lambda: None)
        also[w3.name] = {"tflops": round(w3.flops / r3["per_launch_s"] / 1e12, 3),
                         "frac_of_measured": round(w3.flops / r3["per_launch_s"] / 1e12 / float(peaks.get("bf16_tflops", 1900.0)), 4),
                         "variant": r3["info"]["variant_name"]}
        re = bench_gemm(w, min(args.steps, 100), 5, dev, lambda: None, epilogue_act=_g_act_silu())
        also[w.name + "+bias+silu+residual"] = {
            "tflops": round(w.flops / re["per_launch_s"] / 1e12, 3),
            "us_per_launch": round(re["per_launch_s"] * 1e6, 1),
            "note": "fused epilogue act(A B^T + bias) + residual in the writeback warps"}
        w8 = inputs.WORKLOADS["fp8_8192_e4m3_bf16"]
        r8 = bench_gemm(w8, 100, 10, dev, lambda: None)
        t8 = w8.flops / r8["per_launch_s"] / 1e12
        fp8_peak = 2.0 * float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]))
        also[w8.name] = {"tflops": round(t8, 3), "frac_of_fp8_peak": round(t8 / fp8_peak, 4),
                         "fp8_peak": fp8_peak, "variant": r8["info"]["variant_name"],
                         "peak_note": "measured bf16 burst x 2 (nominal fp8 / bf16 dense ratio 4.5 / 2.25)"}
        wm = inputs.WORKLOADS["mxfp8_8192_e4m3_bf16"]
        rm = bench_gemm(wm, 100, 10, dev, lambda: None)
        tm = wm.flops / rm["per_launch_s"] / 1e12
        also[wm.name] = {"tflops": round(tm, 3), "frac_of_fp8_peak": round(tm / fp8_peak, 4),
                         "fp8_peak": fp8_peak, "variant": rm["info"]["variant_name"],
                         "note": "MX block scaling: UE8M0 scale per 32 K elements, tcgen05.mma kind::mxf8f6f4"}
        w2 = inputs.WORKLOADS["kloop_1024x1024x4096_bf16_bf16"]
        r2 = bench_gemm(w2, 500, 20, dev, lambda: None)
        also[w2.name] = {"tflops": round(w2.flops / r2["per_launch_s"] / 1e12, 3),
                         "us_per_launch": round(r2["per_launch_s"] * 1e6, 2),
                         "variant": r2["info"]["variant_name"], "cluster": r2["info"]["cluster"],
                         "operand_sets": r2["operand_sets"],
                         "note": "32 tiles of 128 x 256: each tile's K split over a cluster of CTAs"}
        w4 = inputs.WORKLOADS["llm_proj_8192x14336x4096_bf16_bf16"]
        r4 = bench_gemm(w4, 50, 5, dev, lambda: None)
        also[w4.name] = {"tflops": round(w4.flops / r4["per_launch_s"] / 1e12, 3),
                         "variant": r4["info"]["variant_name"]}
        hbm = float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]))
        from dense_gemm_blackwell_sm_gb300 import gemm as _g
        for name in ("gemv_m1_n4096_k4096_bf16", "gemv_m8_n4096_k4096_bf16",
                     "gemv_m1_n14336_k4096_bf16", "gemv_m8_n14336_k4096_bf16"):
            g = bench_gemv(inputs.WORKLOADS[name], 200, 20, dev)
            gp = bench_gemv(inputs.WORKLOADS[name], 200, 20, dev, flags=_g.FLAG_STATIC_B)
            also[name] = {"gbs": round(g["gbs"], 1), "frac_of_measured_hbm": round(g["gbs"] / hbm, 4),
                          "frac_of_stated_8000": round(g["gbs"] / STATED_HBM_GBS, 4),
                          "us_per_launch": round(g["us_per_launch"], 2), "variant": g["variant"],
                          "roofline": {"bound": "hbm", "achieved": round(g["gbs"], 1), "peak": hbm, "unit": "GB/s",
                                       "frac": round(g["gbs"] / hbm, 4), "traffic": stored_traffic("gemv", name),
                                       "peak_source": "hbm_gbs %s" % peak_src,
                                       "bytes_per_launch": g["bytes_per_launch"]},
                          "static_b_pdl": {"gbs": round(gp["gbs"], 1), "frac_of_measured_hbm": round(gp["gbs"] / hbm, 4),
                                           "us_per_launch": round(gp["us_per_launch"], 2)},
                          "weight_copies": g["copies"], "timing": "CUDA graph of 200 dependent launches, replayed 3x"}
        line["also"] = also
    if rank == 0 and not args.no_cpu_baseline:
        r = cpu_oracle_rate(w)
        line["cpu_baseline"] = {"value": round(r["tflops"], 6), "unit": "TFLOP/s", "cores": r["threads"],
                                "single_thread": round(r["single_thread_tflops"], 6), "host": r["host"],
                                "kind": "oracle", "sample": r["sample"]}
    if rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
