"""MN-major operands (A stored K x M, B stored K x N) in the step 7-9 kernels,
against the CPU oracle on the logical (K-major) operands."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LAYOUTS = [gemm.LAYOUT_A_MN, gemm.LAYOUT_B_MN, gemm.LAYOUT_A_MN | gemm.LAYOUT_B_MN]
SHAPES = {gemm.S7: (328, 520, 200), gemm.S8: (712, 776, 264), gemm.S9: (1096, 520, 136)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def stored(x: torch.Tensor, mn: bool) -> torch.Tensor:
    return x.t().contiguous() if mn else x.contiguous()


def run(variant, layout, a, b, out):
    M, K = a.shape
    N = b.shape[0]
    plan = gemm.Plan(M, N, K, gemm.dtype_code(a.dtype, out), gemm.make_opts(variant=variant, layout=layout))
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    plan.run(stored(a, bool(layout & gemm.LAYOUT_A_MN)).to(DEV), stored(b, bool(layout & gemm.LAYOUT_B_MN)).to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    return c.double().cpu().numpy()


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ti,to", [("bf16", "bf16"), ("f16", "f32")])
def test_mn_major_integer_bit_exact(variant, layout, ti, to):
    M, N, K = SHAPES[variant]
    a, b = inputs.integer_operands(M, N, K, ti, seed=variant * 10 + layout)
    ref, _ = oracle.gemm(a, b)
    exp = torch.tensor(ref).to(inputs.torch_dtype(to)).double().numpy()
    got = run(variant, layout, a, b, to)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (bad[:3], got[tuple(bad[0])], exp[tuple(bad[0])])


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_mn_major_random_parity(variant, layout):
    M, N, K = SHAPES[variant]
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("normal", 1.0), seed=variant + layout)
    ref, S = oracle.gemm(a, b)
    r = parity.check(run(variant, layout, a, b, "bf16"), ref, S, "bf16")
    assert r["ok"] and r["max_excess_rel"] < 2.0 ** -12, r


def test_auto_plan_with_layout_and_small_m():
    a, b = inputs.make_operands(8, 264, 136, "bf16", ("uniform",), ("uniform",), seed=5)
    ref, S = oracle.gemm(a, b)
    got = run(0, gemm.LAYOUT_A_MN, a, b, "bf16")
    assert parity.check(got, ref, S, "bf16")["ok"]


def test_matmul_reads_transposed_views_in_place():
    a, b = inputs.make_operands(520, 776, 264, "bf16", ("uniform",), ("uniform",), seed=6)
    ref, S = oracle.gemm(a, b)
    at = a.t().contiguous().to(DEV)       # K x M in memory
    bt = b.t().contiguous().to(DEV)       # K x N in memory
    for x, y in ((at.t(), b.to(DEV)), (a.to(DEV), bt.t()), (at.t(), bt.t())):
        c = gemm.matmul(x, y, torch.bfloat16)
        torch.cuda.synchronize()
        assert parity.check(c.double().cpu().numpy(), ref, S, "bf16")["ok"]


def test_layout_argument_checks():
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(100, 64, 64, gemm.BF16_BF16, gemm.make_opts(layout=gemm.LAYOUT_A_MN))
    assert e.value.status == gemm.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(128, 128, 64, gemm.BF16_BF16, gemm.make_opts(variant=gemm.S5, layout=gemm.LAYOUT_B_MN))
    assert e.value.status == gemm.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(128, 128, 64, gemm.BF16_BF16, gemm.make_opts(layout=4))
    assert e.value.status == gemm.ERR_INVALID_ARG
