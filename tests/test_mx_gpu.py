"""GPU parity of the MX block-scaled GEMM (8-bit float operands with one UE8M0
scale per 32 consecutive K elements of every row of A and B, tcgen05.mma
kind::mxf8f6f4 on the step-7 tile, on the step-8 CTA pair and on step 9's two
consumers with 512 x 224 tiles) against the CPU oracle's fp64 block-scaled
product, with the plain and the fused writeback."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# several tiles, ragged M / N, K with a partial 128-element stage and a partial 32-element block
SHAPES = [(300, 520, 272), (1100, 776, 400), (128, 256, 128), (2048, 1024, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run(a, b, sa, sb, out, variant=0, **epi):
    M, K = a.shape
    N = b.shape[0]
    fmt = "mxe4m3" if a.dtype == torch.float8_e4m3fn else "mxe5m2"
    plan = gemm.Plan(M, N, K, gemm.dtype_code(fmt, out), gemm.make_opts(variant=variant))
    info = plan.info()
    ta = inputs.mx_tile_scales(sa, K).to(DEV)
    tb = inputs.mx_tile_scales(sb, K).to(DEV)
    assert ta.numel() == gemm.mx_scale_bytes(M, K) and tb.numel() == gemm.mx_scale_bytes(N, K)
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    plan.run_mx(a.to(DEV), b.to(DEV), c, ta, tb, **epi)
    assert plan.check() == gemm.OK
    plan.destroy()
    return c, info


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_integer_operands_bit_exact(variant, shape, fmt, out):
    # integer operands in [-8, 8] and scales 2^-2 .. 2^2: every term and every
    # fp32 partial sum is exact, so the result is unique
    M, N, K = shape
    a, b = inputs.integer_operands(M, N, K, fmt, seed=M + K, lo=-8, hi=8)
    sa = inputs.mx_scales(M, K, seed=1, e_lo=125, e_hi=129)
    sb = inputs.mx_scales(N, K, seed=2, e_lo=125, e_hi=129)
    c, info = _run(a, b, sa, sb, out, variant)
    assert info["variant"] == variant
    C, _ = oracle.gemm_mx(a, b, sa, sb)
    exp = torch.tensor(C).to(inputs.torch_dtype(out)).double().numpy()
    got = c.double().cpu().numpy()
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (bad[:3], got[tuple(bad[0])], exp[tuple(bad[0])])


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8])
@pytest.mark.parametrize("shape", SHAPES[:3])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_random_parity(variant, shape, fmt):
    M, N, K = shape
    a, b, sa, sb = inputs.mx_operands(M, N, K, fmt, seed=7 + K)
    out = "bf16" if fmt == "e4m3" else "f32"
    c, info = _run(a, b, sa, sb, out, variant)
    C, S = oracle.gemm_mx(a, b, sa, sb)
    r = parity.check(c.double().cpu().numpy(), C, S, out)
    assert r["ok"], (info, r)


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8])
@pytest.mark.parametrize("max_ctas", [1, 3])
def test_few_clusters_many_tiles(variant, max_ctas):
    # few clusters, many tiles each, 21 K blocks a tile: the stage ring and the
    # per-stage TMEM scale slots wrap many times, across tile boundaries
    M, N, K = 1024, 1024, 2688
    a, b = inputs.integer_operands(M, N, K, "e4m3", seed=11, lo=-6, hi=6)
    sa = inputs.mx_scales(M, K, seed=3, e_lo=125, e_hi=129)
    sb = inputs.mx_scales(N, K, seed=4, e_lo=125, e_hi=129)
    plan = gemm.Plan(M, N, K, gemm.dtype_code("mxe4m3", "f32"), gemm.make_opts(variant=variant, max_ctas=max_ctas))
    assert plan.info()["grid"] == max_ctas * plan.info()["cluster"]
    ta, tb = inputs.mx_tile_scales(sa, K).to(DEV), inputs.mx_tile_scales(sb, K).to(DEV)
    c = torch.full((M, N), float("nan"), device=DEV)
    plan.run_mx(a.to(DEV), b.to(DEV), c, ta, tb)
    assert plan.check() == gemm.OK
    plan.destroy()
    C, _ = oracle.gemm_mx(a, b, sa, sb)
    bad = np.argwhere(c.double().cpu().numpy() != C)
    assert bad.size == 0, bad[:3]


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8])
def test_scales_only_touch_their_own_block(variant):
    # one scale byte of A and one of B changed: only that row and that column move
    M, N, K = 512, 512, 256
    a, b = inputs.integer_operands(M, N, K, "e4m3", seed=5, lo=-4, hi=4)
    sa = torch.full((M, K // 32), 127, dtype=torch.uint8)
    sb = torch.full((N, K // 32), 127, dtype=torch.uint8)
    sa[77, 5] = 130
    sb[200, 2] = 124
    c, _ = _run(a, b, sa, sb, "f32", variant)
    C, _ = oracle.gemm_mx(a, b, sa, sb)
    assert np.array_equal(c.double().cpu().numpy(), C)
    C0, _ = oracle.gemm(a, b)
    diff = np.argwhere(C != C0)
    assert ((diff[:, 0] == 77) | (diff[:, 1] == 200)).all()
    assert (diff[:, 0] == 77).any() and (diff[:, 1] == 200).any()


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8])
@pytest.mark.parametrize("act", [gemm.ACT_NONE, gemm.ACT_RELU, gemm.ACT_SILU, gemm.ACT_GELU_ERF])
def test_fused_epilogue(variant, act):
    M, N, K = 700, 776, 336
    out = "bf16" if act % 2 else "f32"
    a, b, sa, sb = inputs.mx_operands(M, N, K, "e4m3", seed=40 + act)
    g = torch.Generator().manual_seed(act)
    bias = torch.randn(N, generator=g).float()
    res = torch.randn(M, N, generator=g).to(inputs.torch_dtype(out))
    rs = (torch.rand(M, generator=g) + 0.5).float()
    c, _ = _run(a, b, sa, sb, out, variant, bias=bias.to(DEV), residual=res.to(DEV), act=act,
                scale_a=rs.to(DEV))
    C, S = oracle.gemm_mx(a, b, sa, sb)
    ref = oracle.epilogue(C, bias, res, act, scale_a=rs)
    pre = oracle.epilogue(C, bias, None, oracle.ACT_NONE, scale_a=rs)
    r = parity.check_epilogue(c.double().cpu().numpy(), ref, pre, oracle.scale(S, rs), np.abs(res.double().numpy()),
                              out, act)
    assert r["ok"], r


def test_large_sampled_rows():
    M = N = K = 4096
    a, b, sa, sb = inputs.mx_operands(M, N, K, "e4m3", seed=3)
    c, info = _run(a, b, sa, sb, "bf16")
    rows = [0, 127, 128, 1000, 2047, 2048, 4095]
    C, S = oracle.gemm_mx(a, b, sa, sb, rows=rows)
    r = parity.check(c[rows].double().cpu().numpy(), C, S, "bf16")
    assert r["ok"], (info, r)
    assert bool(torch.isfinite(c).all())


def test_rejections():
    M = N = K = 256
    a = torch.zeros(M, K, dtype=torch.float8_e4m3fn, device=DEV)
    s = torch.full((gemm.mx_scale_bytes(M, K),), 127, dtype=torch.uint8, device=DEV)
    c = torch.zeros(M, N, device=DEV)
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(M, N, K, gemm.MXE4M3_F32, gemm.make_opts(variant=gemm.S9))
    assert e.value.status == gemm.ERR_UNSUPPORTED_SHAPE
    plan = gemm.Plan(M, N, K, gemm.MXE4M3_F32)
    with pytest.raises(gemm.GemmError) as e:
        plan.run(a, a, c)        # no scales
    assert e.value.status == gemm.ERR_INVALID_ARG
    with pytest.raises(gemm.GemmError) as e:
        plan.run_epilogue(a, a, c, act=gemm.ACT_RELU)
    assert e.value.status == gemm.ERR_INVALID_ARG
    with pytest.raises(gemm.GemmError) as e:
        plan.run_mx(a, a, c, s[1:], s)
    assert e.value.status == gemm.ERR_MISALIGNED
    plan.run_mx(a, a, c, s, s)
    assert plan.check() == gemm.OK and bool((c == 0).all())
    plan.destroy()
    p2 = gemm.Plan(M, N, K, gemm.E4M3_F32)
    with pytest.raises(gemm.GemmError) as e:
        p2.run_mx(a, a, c, s, s)
    assert e.value.status == gemm.ERR_UNSUPPORTED_DTYPE
    p2.destroy()


# step 9: 224-column tiles start B's rows at a multiple of 32 but not of 128, so
# each tile's B scales are regrouped from three 128-row blocks; N spans several
# tile columns (tn = 0..8 covers every offset of a tile inside a 128-row block),
# M several tile rows, K a partial 128-element stage
S9_SHAPES = [(1100, 2000, 400), (512, 224, 128), (300, 520, 272), (4096, 8192, 1024)]


@pytest.mark.parametrize("shape", S9_SHAPES)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_step9_integer_operands_bit_exact(shape, fmt):
    M, N, K = shape
    a, b = inputs.integer_operands(M, N, K, fmt, seed=M + 3 * K, lo=-8, hi=8)
    sa = inputs.mx_scales(M, K, seed=5, e_lo=125, e_hi=129)
    sb = inputs.mx_scales(N, K, seed=6, e_lo=125, e_hi=129)
    c, info = _run(a, b, sa, sb, "bf16", gemm.S9)
    assert info["variant"] == gemm.S9 and info["tile_n"] == 224 and info["consumers"] == 2
    C, _ = oracle.gemm_mx(a, b, sa, sb)
    exp = torch.tensor(C).to(torch.bfloat16).double().numpy()
    bad = np.argwhere(c.double().cpu().numpy() != exp)
    assert bad.size == 0, bad[:3]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_step9_random_parity(fmt):
    M, N, K = 1100, 2000, 400
    a, b, sa, sb = inputs.mx_operands(M, N, K, fmt, seed=17)
    c, info = _run(a, b, sa, sb, "bf16", gemm.S9)
    C, S = oracle.gemm_mx(a, b, sa, sb)
    r = parity.check(c.double().cpu().numpy(), C, S, "bf16")
    assert r["ok"], (info, r)


def test_step9_scales_only_touch_their_own_block():
    # B rows 200 (tile 0, second regrouped block) and 300 (tile 1, which starts at
    # row 224 inside the second 128-row block): only their columns move
    M, N, K = 512, 896, 256
    a, b = inputs.integer_operands(M, N, K, "e4m3", seed=9, lo=-4, hi=4)
    sa = torch.full((M, K // 32), 127, dtype=torch.uint8)
    sb = torch.full((N, K // 32), 127, dtype=torch.uint8)
    sa[77, 5] = 130
    sb[200, 2] = 124
    sb[300, 7] = 129
    c, _ = _run(a, b, sa, sb, "bf16", gemm.S9)
    C, _ = oracle.gemm_mx(a, b, sa, sb)
    assert np.array_equal(c.double().cpu().numpy(), torch.tensor(C).to(torch.bfloat16).double().numpy())
    C0, _ = oracle.gemm(a, b)
    diff = np.argwhere(C != C0)
    assert ((diff[:, 0] == 77) | (diff[:, 1] == 200) | (diff[:, 1] == 300)).all()
    assert (diff[:, 1] == 200).any() and (diff[:, 1] == 300).any()


def test_step9_plan_with_fused_epilogue():
    # a step-9 block-scaled plan runs its fused epilogue on step 8's tile
    M, N, K = 700, 776, 336
    a, b, sa, sb = inputs.mx_operands(M, N, K, "e4m3", seed=41)
    g = torch.Generator().manual_seed(1)
    bias = torch.randn(N, generator=g).float()
    res = torch.randn(M, N, generator=g).to(torch.bfloat16)
    c, info = _run(a, b, sa, sb, "bf16", gemm.S9, bias=bias.to(DEV), residual=res.to(DEV), act=gemm.ACT_SILU)
    assert info["variant"] == gemm.S9
    C, S = oracle.gemm_mx(a, b, sa, sb)
    ref = oracle.epilogue(C, bias, res, gemm.ACT_SILU)
    pre = oracle.epilogue(C, bias, None, oracle.ACT_NONE)
    r = parity.check_epilogue(c.double().cpu().numpy(), ref, pre, S, np.abs(res.double().numpy()), "bf16",
                              gemm.ACT_SILU)
    assert r["ok"], r


def test_bench_workload_sampled_rows():
    # the 8192^3 block-scaled workload the bench times, in its launch configuration
    w = inputs.WORKLOADS["mxfp8_8192_e4m3_bf16"]
    a, b = inputs.workload_operands(w)
    sa, sb = inputs.workload_mx_scales(w)
    c, info = _run(a, b, sa, sb, w.out_dtype)
    rows = [0, 1, 127, 128, 4095, 4096, 8191] + list(range(1000, 8192, 1777))
    C, S = oracle.gemm_mx(a, b, sa, sb, rows=rows)
    r = parity.check(c[rows].double().cpu().numpy(), C, S, w.out_dtype)
    assert r["ok"], (info, r)
    assert bool(torch.isfinite(c).all())
