"""Host-side logic of bench.py: peaks, traffic bookkeeping, the max-over-ranks
aggregation across world_size-2 gloo processes, and the single JSON line of
the reference arm under torchrun (no GPU needed)."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_aggregate_takes_the_slowest_rank_and_counts_all_work():
    t, rate = bench.aggregate([0.5, 0.8, 0.6], 100.0)
    assert t == 0.8
    assert rate == pytest.approx(300.0 / 0.8)


def test_peaks_and_traffic_lookup():
    peaks, src = bench.measured_peaks()
    assert src in ("measured", "fallback")
    assert peaks["bf16_tflops"] > 0 and peaks["hbm_gbs"] > 0
    assert len(bench.source_hash("ws")) == 16
    assert bench.stored_traffic("ws", "no_such_workload") is None


def test_traffic_key_ignores_comments_and_layout_only():
    a = "int f(int x) {  // doubles\n  return 2 * x; /* twice */ }\n"
    b = "int f(int x) {\n\treturn 2 * x;\n}"
    c = "int f(int x) { return 3 * x; }"
    assert bench.code_tokens(a) == bench.code_tokens(b) == "int f(int x) { return 2 * x; }"
    assert bench.code_tokens(c) != bench.code_tokens(a)
    # every stored capture carries the key of the code it was taken on
    import json
    with open(bench.TRAFFIC_FILE) as f:
        d = json.load(f)
    for kind in ("ws", "mx", "gemv"):
        assert all(len(e["source_hash"]) == 16 for e in d[kind].values())


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, ws, local, barrier, gather = bench._dist()
    barrier()
    times = gather(0.25 * (r + 1))
    barrier()
    q.put((r, ws, times))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_gloo_gather_and_aggregate():
    if torch.cuda.is_available():
        pytest.skip("the CPU (gloo) path is exercised on hosts without a GPU")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, ws, times in out:
        assert ws == 2 and times == [0.25, 0.5]
    t, rate = bench.aggregate(out[0][2], 10.0)
    assert t == 0.5 and rate == pytest.approx(40.0)


def test_reference_arm_prints_one_line_under_torchrun():
    if torch.cuda.is_available():
        pytest.skip("the CPU (gloo) path is exercised on hosts without a GPU")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--workload", "single_tile_128x128x64_f16_f32"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["ms_per_step"] > 0 and d["higher_is_better"] is True and d["config"]["workload"] == \
        "single_tile_128x128x64_f16_f32"


def test_reference_arm_steps_fit_the_run():
    """--impl reference reports the steps it ran: steps x ms_per_step is the
    time of its timed steps, inside the wall time of the whole run."""
    if torch.cuda.is_available():
        pytest.skip("the CPU path is exercised on hosts without a GPU")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "4", "--warmup", "3",
           "--workload", "kloop_1024x1024x4096_bf16_bf16"]
    t0 = time.time()
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    wall = time.time() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert d["steps"] == 4
    timed = d["steps"] * d["ms_per_step"] / 1e3
    assert 0 < timed < wall
    rows = d["config"]["rows_per_step"]
    assert 1 <= rows <= 1024
    # the value is the rate of the sampled work
    assert d["value"] == pytest.approx(2.0 * rows * 1024 * 4096 * d["steps"] / timed / 1e12, rel=1e-3)
    host = d["cpu_baseline"]["host"]
    assert host["affinity_cores"] >= 1 and host["model"]


def test_clock_sampler_windows_and_load():
    """Samples are matched to a timed window by nvidia-smi's timestamp, and a
    sample counts as under load above 40 % of the power limit."""
    lines = ["2026/12/03 05:00:00.000, 0, 1000, 2070, 300.0, 1400.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/03 05:00:00.050, 0, 1900, 2070, 1300.0, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
             "2026/12/03 05:00:00.100, 0, 1800, 2070, 1350.0, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
             "2026/12/03 05:00:02.000, 0, 900, 2070, 250.0, 1400.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    c = bench.ClockSampler(0)
    c.lines = lines
    smp = c.parse(lines)
    t = smp[0]["t"]
    assert smp[1]["t"] - t == pytest.approx(0.05, abs=1e-6)
    s = c.summary(t + 0.1, t + 0.11)   # the window is widened by half a sample period on each side
    assert s["samples"] == 2 and s["samples_under_load"] == 2 and s["sm_mhz_under_load"] in (1800.0, 1900.0)
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1350.0
    a = c.summary()
    assert a["samples"] == 4 and a["samples_under_load"] == 2 and a["sm_max_mhz"] == 2070.0
    # with instantaneous power sampled, it decides load: the averaged draw lags a
    # short timed region
    inst = ["2026/12/03 05:00:00.000, 0, 2070, 2070, 120.0, 1400.0, 0x0, Not Active, Not Active, Not Active, Not Active, 160.0",
            "2026/12/03 05:00:00.050, 0, 2070, 2070, 177.6, 1400.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1223.3",
            "2026/12/03 05:00:00.100, 0, 1620, 2070, 307.8, 1400.0, 0x4, Not Active, Not Active, Not Active, Active, 1391.2",
            "2026/12/03 05:00:00.150, 0, 2070, 2070, 324.6, 1400.0, 0x0, Not Active, Not Active, Not Active, Not Active, [N/A]"]
    c.lines = inst
    b = c.summary()
    assert b["samples"] == 4 and b["samples_under_load"] == 2 and b["power_w_instant_max"] == 1391.2
    assert b["power_w_max"] == 324.6 and b["sm_mhz_under_load"] in (1620.0, 2070.0)
