"""GPU parity of the 8-bit float GEMM (E4M3 / E5M2 inputs, fp32 accumulation
in Tensor Memory, fp32 or bf16 output) of the warp-specialised kernels
(variants 7-9, tcgen05.mma kind::f8f6f4) against the CPU oracle, including the
fused epilogue with per-row / per-column dequantisation scales."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMTS = ["e4m3", "e5m2"]
# ragged in M, N and K (K = 128-byte boxes plus a 16-byte tail) and several tiles
SHAPES = {gemm.S7: (300, 520, 272), gemm.S8: (700, 776, 400), gemm.S9: (1100, 520, 144)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _plan_run(variant, a, b, out):
    M, K = a.shape
    N = b.shape[0]
    plan = gemm.Plan(M, N, K, gemm.dtype_code(a.dtype, out), gemm.make_opts(variant=variant))
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    info = plan.info()
    plan.destroy()
    return c, info


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_integer_operands_bit_exact(variant, fmt, out):
    # integers in [-8, 8] are exact in both formats; partial sums stay below 2^16
    M, N, K = SHAPES[variant]
    a, b = inputs.integer_operands(M, N, K, fmt, seed=variant, lo=-8, hi=8)
    c, info = _plan_run(variant, a, b, out)
    assert info["variant"] == variant
    C, _ = oracle.gemm(a, b)
    exp = torch.tensor(C).to(inputs.torch_dtype(out)).double().numpy()
    got = c.double().cpu().numpy()
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (bad[:3], got[tuple(bad[0])], exp[tuple(bad[0])])


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("fmt", FMTS)
def test_random_parity(variant, fmt):
    M, N, K = SHAPES[variant]
    out = "bf16" if variant == gemm.S8 else "f32"
    a, b = inputs.make_operands(M, N, K, fmt, ("normal", 1.0), ("uniform",), seed=17 + variant)
    c, info = _plan_run(variant, a, b, out)
    C, S = oracle.gemm(a, b)
    r = parity.check(c.double().cpu().numpy(), C, S, out)
    assert r["ok"], (info, r)


def test_automatic_plan_and_matmul():
    M, N, K = 520, 1032, 336
    a, b = inputs.make_operands(M, N, K, "e4m3", ("uniform",), ("normal", 1.0), seed=5)
    da, db = a.to(DEV), b.to(DEV)
    plan = gemm.Plan(M, N, K, gemm.E4M3_F32)
    assert plan.info()["variant"] in (gemm.S7, gemm.S8, gemm.S9)
    plan.destroy()
    c = gemm.matmul(da, db)
    c2 = gemm.matmul(da.t().contiguous().t(), db, out_dtype=torch.bfloat16)   # strided view: copied
    torch.cuda.synchronize()
    C, S = oracle.gemm(a, b)
    assert parity.check(c.double().cpu().numpy(), C, S, "f32")["ok"]
    assert parity.check(c2.double().cpu().numpy(), C, S, "bf16")["ok"]


def test_large_sampled_rows():
    M = N = K = 4096
    a, b = inputs.make_operands(M, N, K, "e4m3", ("uniform",), ("normal", 1.0), seed=11)
    c, info = _plan_run(gemm.VARIANT_AUTO, a, b, "bf16")
    rows = [0, 127, 128, 255, 256, 511, 512, 2047, 2048, 4095]
    C, S = oracle.gemm_rows(a, b, rows)
    r = parity.check(c[rows].double().cpu().numpy(), C, S, "bf16")
    assert r["ok"], (info, r)
    assert bool(torch.isfinite(c).all())


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("act", [gemm.ACT_NONE, gemm.ACT_RELU, gemm.ACT_SILU, gemm.ACT_GELU_TANH])
def test_scaled_epilogue(variant, act):
    M, N, K = SHAPES[variant]
    fmt = "e4m3" if act % 2 == 0 else "e5m2"
    out = "bf16" if (act + variant) % 2 else "f32"
    a, b = inputs.make_operands(M, N, K, fmt, ("normal", 1.0), ("uniform",), seed=31 * act + variant)
    g = torch.Generator().manual_seed(act + 10 * variant)
    sa = (torch.rand(M, generator=g) * 0.5 + 0.25).float()
    sb = (torch.rand(N, generator=g) * 0.5 + 0.25).float()
    bias = torch.randn(N, generator=g).float()
    res = (torch.randn(M, N, generator=g)).to(inputs.torch_dtype(out))
    plan = gemm.Plan(M, N, K, gemm.dtype_code(a.dtype, out), gemm.make_opts(variant=variant))
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    plan.run_epilogue(a.to(DEV), b.to(DEV), c, bias=bias.to(DEV), residual=res.to(DEV), act=act,
                      scale_a=sa.to(DEV), scale_b=sb.to(DEV))
    assert plan.check() == gemm.OK
    plan.destroy()
    C, S = oracle.gemm(a, b)
    ref = oracle.epilogue(C, bias, res, act, scale_a=sa, scale_b=sb)
    pre = oracle.epilogue(C, bias, None, oracle.ACT_NONE, scale_a=sa, scale_b=sb)
    S_scaled = oracle.scale(S, sa, sb)   # the scales are positive
    r = parity.check_epilogue(c.double().cpu().numpy(), ref, pre, S_scaled, np.abs(res.double().numpy()), out, act)
    assert r["ok"], r


def test_scales_alone_on_16bit_inputs():
    # the scale terms are not specific to 8-bit inputs
    M, N, K = 384, 264, 128
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=3)
    sa = torch.full((M,), 0.5)
    sb = 2.0 ** torch.randint(-3, 4, (N,), generator=torch.Generator().manual_seed(1)).float()
    plan = gemm.Plan(M, N, K, gemm.BF16_F32, gemm.make_opts(variant=gemm.S8))
    c = torch.empty((M, N), device=DEV)
    plan.run_epilogue(a.to(DEV), b.to(DEV), c, scale_a=sa.to(DEV), scale_b=sb.to(DEV))
    assert plan.check() == gemm.OK
    plan.destroy()
    C, _ = oracle.gemm(a, b)
    assert np.array_equal(c.double().cpu().numpy(), oracle.scale(C, sa, sb))


def test_host_entry_point():
    M, N, K = 256, 512, 256
    a, b = inputs.make_operands(M, N, K, "e5m2", ("uniform",), ("normal", 1.0), seed=2)
    ah, bh = a.view(torch.uint8).pin_memory(), b.view(torch.uint8).pin_memory()
    ch = torch.empty((M, N), dtype=torch.float32).pin_memory()
    da = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    db = torch.empty((N, K), dtype=torch.uint8, device=DEV)
    dc = torch.empty((M, N), dtype=torch.float32, device=DEV)
    st = gemm.gemm_run_host(M, N, K, ah.data_ptr(), bh.data_ptr(), ch.data_ptr(), gemm.E5M2_F32,
                            da.data_ptr(), db.data_ptr(), dc.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert st == gemm.OK
    torch.cuda.synchronize()
    C, S = oracle.gemm(a, b)
    assert parity.check(ch.double().numpy(), C, S, "f32")["ok"]


def test_rejections():
    a = torch.zeros(64, 64, dtype=torch.float8_e4m3fn, device=DEV)
    c = torch.full((64, 64), 1.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(64, 64, 64, gemm.E4M3_F32, gemm.make_opts(variant=gemm.S6))
    assert e.value.status == gemm.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(gemm.GemmError):
        gemm.Plan(64, 64, 64, gemm.E4M3_F32, gemm.make_opts(variant=gemm.S8, layout=gemm.LAYOUT_B_MN))
    with pytest.raises(gemm.GemmError):
        gemm.Plan(64, 64, 40, gemm.E4M3_F32)
    assert gemm.gemm_run(64, 64, 64, a.data_ptr(), a.data_ptr(), c.data_ptr(), gemm.E4M3_BF16,
                         torch.cuda.current_stream().cuda_stream) == gemm.OK
    torch.cuda.synchronize()
    assert bool((c == 0).all())


# stream-K with 8-bit operands: tiles outnumber the resident clusters and are split
# between clusters (K blocks of 128 elements here)
SK_SHAPES = {gemm.S7: (1280, 4352, 528), gemm.S8: (1280, 4352, 272), gemm.S9: (2560, 4352, 144)}


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_stream_k_integer_bit_exact(variant, out):
    M, N, K = SK_SHAPES[variant]
    a, b = inputs.integer_operands(M, N, K, "e4m3", seed=50 + variant, lo=-8, hi=8)
    plan = gemm.Plan(M, N, K, gemm.dtype_code("e4m3", out), gemm.make_opts(variant=variant, sched=gemm.SCHED_STREAM_K))
    info = plan.info()
    assert info["sched"] == gemm.SCHED_STREAM_K and info["tiles"] > info["grid"] // info["cluster"]
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    for _ in range(2):
        c.fill_(float("nan"))
        plan.run(a.to(DEV), b.to(DEV), c)
        assert plan.check() == gemm.OK
    plan.destroy()
    C, _ = oracle.gemm(a, b)
    exp = torch.tensor(C).to(inputs.torch_dtype(out)).double().numpy()
    bad = np.argwhere(c.double().cpu().numpy() != exp)
    assert bad.size == 0, (info, bad[:3])


@pytest.mark.parametrize("M,N,K,split", [(1024, 1024, 4096, 0), (300, 520, 1296, 3)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_split_k_cluster_integer_bit_exact(M, N, K, split, out):
    a, b = inputs.integer_operands(M, N, K, "e5m2", seed=60 + split, lo=-4, hi=4)
    opts = gemm.make_opts(variant=gemm.S7 if split else 0, split_k=split)
    plan = gemm.Plan(M, N, K, gemm.dtype_code("e5m2", out), opts)
    info = plan.info()
    if split:
        assert info["variant"] == gemm.S7 and info["cluster"] == split, info
    else:  # 32 K blocks: two slices, of step 8's pair tiles (as many SMs as step 7's)
        assert (info["variant"], info["cluster"]) == (gemm.S8, 4), info
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    C, _ = oracle.gemm(a, b)
    exp = torch.tensor(C).to(inputs.torch_dtype(out)).double().numpy()
    bad = np.argwhere(c.double().cpu().numpy() != exp)
    assert bad.size == 0, (info, bad[:3])
