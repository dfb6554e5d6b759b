"""GPU parity of the fused writeback epilogue, C = act(A B^T + bias) + residual,
of the step 7-9 kernels against the CPU oracle's fp64 epilogue."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ACTS = [gemm.ACT_NONE, gemm.ACT_RELU, gemm.ACT_SILU, gemm.ACT_GELU_TANH, gemm.ACT_GELU_ERF]
SHAPES = {gemm.S7: (300, 520, 200), gemm.S8: (700, 776, 264), gemm.S9: (1100, 520, 136)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run(variant, a, b, out, bias, residual, act, alias=False):
    M, K = a.shape
    N = b.shape[0]
    plan = gemm.Plan(M, N, K, gemm.dtype_code(a.dtype, out), gemm.make_opts(variant=variant))
    t = inputs.torch_dtype(out)
    if alias:
        c = residual.to(DEV).clone()
        res = c
    else:
        c = torch.full((M, N), float("nan"), device=DEV, dtype=t)
        res = None if residual is None else residual.to(DEV)
    plan.run_epilogue(a.to(DEV), b.to(DEV), c, bias=None if bias is None else bias.to(DEV), residual=res, act=act)
    assert plan.check() == gemm.OK
    plan.destroy()
    return c.double().cpu().numpy()


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_integer_relu_bias_residual_bit_exact(variant, out):
    M, N, K = SHAPES[variant]
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=variant)
    g = torch.Generator().manual_seed(variant)
    bias = torch.randint(-20, 21, (N,), generator=g).float()
    res = torch.randint(-8, 9, (M, N), generator=g).to(inputs.torch_dtype(out))
    C, _ = oracle.gemm(a, b)
    ref = oracle.epilogue(C, bias, res, oracle.ACT_RELU)
    exp = torch.tensor(ref).to(inputs.torch_dtype(out)).double().numpy()
    got = _run(variant, a, b, out, bias, res, gemm.ACT_RELU)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (bad[:3], got[tuple(bad[0])], exp[tuple(bad[0])])


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("use_bias,use_res", [(True, True), (True, False), (False, True)])
def test_random_epilogue_parity(variant, act, use_bias, use_res):
    M, N, K = SHAPES[variant]
    out = "bf16" if (act + variant) % 2 else "f32"
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("normal", 0.2), seed=act * 7 + variant)
    g = torch.Generator().manual_seed(act + 100 * variant)
    bias = (torch.randn(N, generator=g) * 2).float() if use_bias else None
    res = (torch.randn(M, N, generator=g) * 3).to(inputs.torch_dtype(out)) if use_res else None
    C, S = oracle.gemm(a, b)
    ref = oracle.epilogue(C, bias, res, act)
    pre = C + (bias.double().numpy()[None, :] if use_bias else 0.0)
    res_abs = np.abs(res.double().numpy()) if use_res else np.zeros_like(C)
    got = _run(variant, a, b, out, bias, res, act)
    r = parity.check_epilogue(got, ref, pre, S, res_abs, out, act)
    assert r["ok"], r


@pytest.mark.parametrize("variant", [gemm.S8, gemm.S9])
def test_residual_may_be_the_output(variant):
    M, N, K = SHAPES[variant]
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("uniform",), seed=31)
    res = (torch.randn(M, N, generator=torch.Generator().manual_seed(31))).to(torch.bfloat16)
    C, S = oracle.gemm(a, b)
    ref = oracle.epilogue(C, None, res, gemm.ACT_SILU)
    got = _run(variant, a, b, "bf16", None, res, gemm.ACT_SILU, alias=True)
    assert parity.check_epilogue(got, ref, C, S, np.abs(res.double().numpy()), "bf16", gemm.ACT_SILU)["ok"]


def test_epilogue_argument_checks():
    a = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    c = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    gv = gemm.Plan(8, 64, 64, gemm.BF16_BF16, gemm.make_opts(variant=gemm.GEMV))
    with pytest.raises(gemm.GemmError) as e:
        gv.run_epilogue(a[:8], a, c[:8], act=gemm.ACT_RELU)
    assert e.value.status == gemm.ERR_UNSUPPORTED_SHAPE
    ws = gemm.Plan(64, 64, 64, gemm.BF16_BF16, gemm.make_opts(variant=gemm.S8))
    with pytest.raises(gemm.GemmError) as e:
        ws.run_epilogue(a, a, c, act=9)
    assert e.value.status == gemm.ERR_INVALID_ARG
    flat = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gemm.GemmError) as e:
        ws.run_epilogue(a, a, c, residual=flat[1:], act=gemm.ACT_NONE)
    assert e.value.status == gemm.ERR_MISALIGNED
    gv.destroy()
    ws.destroy()


ACT_SWEEP = np.concatenate([np.linspace(-20.0, 20.0, 3001), -np.logspace(-30, 4, 200), np.logspace(-30, 4, 200),
                            [0.0, -88.0, -87.0, 88.0, 89.0, -1e4, 1e4]]).astype(np.float32)


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("act", [gemm.ACT_RELU, gemm.ACT_SILU, gemm.ACT_GELU_TANH, gemm.ACT_GELU_ERF])
def test_activation_over_its_range(variant, out, act):
    """With A = B = 0 every row of C is act(bias): the activation alone, over a
    dense sweep of [-20, 20], magnitudes from 1e-30 to 1e4 of both signs, and the
    points where e^x leaves fp32's range.  fp32 C stays within 2^-20 |x| of the
    fp64 value (plus its own rounding); bf16 C within the parity bound."""
    N = ACT_SWEEP.size
    N += (-N) % 8
    bias = np.zeros(N, dtype=np.float32)
    bias[:ACT_SWEEP.size] = ACT_SWEEP
    M, K = 130, 64
    a = torch.zeros(M, K, dtype=torch.bfloat16)
    b = torch.zeros(N, K, dtype=torch.bfloat16)
    got = _run(variant, a, b, out, torch.from_numpy(bias), None, act)
    ref = oracle.epilogue(np.zeros((M, N)), bias, None, act)
    pre = np.broadcast_to(bias.astype(np.float64), (M, N))
    r = parity.check_epilogue(got, ref, pre, np.zeros((M, N)), np.zeros((M, N)), out, act)
    assert r["ok"], r
    if out == "f32":
        err = np.abs(got - ref)
        lim = 2.0 ** -20 * np.abs(pre) + 2.0 ** -24 * np.abs(ref)
        worst = np.unravel_index(np.argmax(err - lim), err.shape)
        assert (err <= lim).all(), (pre[worst], got[worst], ref[worst])


@pytest.mark.parametrize("out,act,alias", [("bf16", gemm.ACT_RELU, False), ("bf16", gemm.ACT_RELU, True),
                                           ("f32", gemm.ACT_NONE, False)])
def test_step9_epilogue_with_32_byte_rows(out, act, alias):
    """N a multiple of 16 and 32-byte aligned rows: step 9's fused writeback then
    reads the residual and writes C 32 bytes per lane and access.  Integer inputs,
    bias and residual: bit-exact, including the last, ragged row tile and the
    residual given as C itself."""
    M, N, K = 1040, 2064, 200
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=77)
    g = torch.Generator().manual_seed(77)
    bias = torch.randint(-20, 21, (N,), generator=g).float()
    res = torch.randint(-8, 9, (M, N), generator=g).to(inputs.torch_dtype(out))
    C, _ = oracle.gemm(a, b)
    exp = torch.tensor(oracle.epilogue(C, bias, res, act)).to(inputs.torch_dtype(out)).double().numpy()
    got = _run(gemm.S9, a, b, out, bias, res, act, alias=alias)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (bad[:3], got[tuple(bad[0])], exp[tuple(bad[0])])
