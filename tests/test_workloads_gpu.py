"""Parity at the workloads' full sizes, in the launch configuration the bench
times (the automatic plan), against the CPU oracle.

Small workloads (the single tile, the K-loop 1024^2 x 4096 GEMM and the decode
GEMVs) are compared element by element in full.  For the 4096^3, 8192^3 and
8192 x 14336 x 4096 GEMMs the oracle computes a stated row sample: the first
and last rows, rows on both sides of the 128-, 256- and 512-row tile
boundaries, and seeded random rows, each against all N columns.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

FULL = ["single_tile_128x128x64_f16_f32", "kloop_1024x1024x4096_bf16_bf16",
        "gemv_m1_n4096_k4096_bf16", "gemv_m8_n4096_k4096_bf16",
        "gemv_m1_n14336_k4096_bf16", "gemv_m8_n14336_k4096_bf16"]
SAMPLED = ["square_4096_f16_f32", "large_8192_bf16_bf16", "llm_proj_8192x14336x4096_bf16_bf16",
           "fp8_8192_e4m3_bf16"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def sample_rows(M: int, seed: int = 0) -> list[int]:
    rows = {0, M - 1}
    for t in (128, 256, 512):
        for b in range(t, M, t * 7):
            rows.update((b - 1, b))
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, M, 8))
    return sorted(r for r in rows if 0 <= r < M)


def run_auto(w: inputs.Workload, a, b, variant: int = 0):
    code = gemm.dtype_code(w.in_dtype, w.out_dtype)
    plan = gemm.Plan(w.M, w.N, w.K, code, gemm.make_opts(variant=variant))
    c = torch.full((w.M, w.N), float("nan"), device=DEV, dtype=inputs.torch_dtype(w.out_dtype))
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    info = plan.info()
    plan.destroy()
    return c, info


@pytest.mark.parametrize("name", FULL)
def test_workload_full_parity(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.workload_operands(w)
    c, info = run_auto(w, a, b)
    ref, S = oracle.gemm(a, b)
    r = parity.check(c.float().cpu().numpy(), ref, S, w.out_dtype)
    assert r["ok"], (info, r)
    assert r["max_excess_rel"] < 2.0 ** -12, (info, r)


@pytest.mark.parametrize("name", SAMPLED)
def test_workload_sampled_parity(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.workload_operands(w)
    c, info = run_auto(w, a, b)
    rows = sample_rows(w.M)
    ref, S = oracle.gemm_rows(a, b, rows)
    got = c[rows].float().cpu().numpy()
    r = parity.check(got, ref, S, w.out_dtype)
    assert r["ok"], (info, r)
    assert r["max_excess_rel"] < 2.0 ** -12, (info, r)
    # every element is finite (no unwritten tile anywhere)
    assert bool(torch.isfinite(c).all())


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
def test_large_workload_every_pair_kernel(variant):
    w = inputs.WORKLOADS["large_8192_bf16_bf16"]
    a, b = inputs.workload_operands(w)
    c, info = run_auto(w, a, b, variant)
    rows = sample_rows(w.M, seed=variant)
    ref, S = oracle.gemm_rows(a, b, rows)
    r = parity.check(c[rows].float().cpu().numpy(), ref, S, w.out_dtype)
    assert r["ok"], (info, r)
    assert bool(torch.isfinite(c).all())


@pytest.mark.parametrize("variant", [gemm.GEMV, gemm.GEMV_TC])
def test_gemv_workloads_both_kernels(variant):
    for name in ("gemv_m1_n4096_k4096_bf16", "gemv_m8_n14336_k4096_bf16"):
        w = inputs.WORKLOADS[name]
        a, b = inputs.workload_operands(w)
        c, info = run_auto(w, a, b, variant)
        ref, S = oracle.gemm(a, b)
        r = parity.check(c.float().cpu().numpy(), ref, S, w.out_dtype)
        assert r["ok"], (name, info, r)
