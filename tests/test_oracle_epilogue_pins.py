"""Pins of the oracle's fused epilogue, act(C + bias[col]) + residual (no GPU).

Checked against things other than itself: special values, the odd-part
identity f(x) - f(-x) = x that SiLU and both GeLU forms satisfy, PyTorch's own
fp64 activations (a separate implementation), exact integer bias / residual
arithmetic, and the slope bounds the parity rule relies on.  Planted mistakes
(bias added per row, residual added before the activation, one activation
swapped for another) must fail a pin.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import parity

ACTS = [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_SILU, oracle.ACT_GELU_TANH, oracle.ACT_GELU_ERF]


def torch_act(x: np.ndarray, act: int) -> np.ndarray:
    t = torch.tensor(x, dtype=torch.float64)
    if act == oracle.ACT_RELU:
        t = F.relu(t)
    elif act == oracle.ACT_SILU:
        t = F.silu(t)
    elif act == oracle.ACT_GELU_TANH:
        t = F.gelu(t, approximate="tanh")
    elif act == oracle.ACT_GELU_ERF:
        t = F.gelu(t)
    return t.numpy()


def real_epilogue(C, bias, residual, act):
    return oracle.epilogue(C, bias=bias, residual=residual, act=act)


# ---------------------------------------------------------------- pins

def pin_special_values(fn) -> bool:
    for act in ACTS:
        if fn(np.zeros((1, 1)), None, None, act)[0, 0] != 0.0:
            return False
    big = np.array([[30.0, -30.0]])
    silu = fn(big, None, None, oracle.ACT_SILU)[0]
    relu = fn(big, None, None, oracle.ACT_RELU)[0]
    return abs(silu[0] - 30.0) < 1e-9 and abs(silu[1]) < 1e-9 and relu[0] == 30.0 and relu[1] == 0.0


def pin_odd_part(fn) -> bool:
    """silu(x) - silu(-x) = x and gelu(x) - gelu(-x) = x (both forms)."""
    x = np.linspace(-6, 6, 97).reshape(1, -1)
    for act in (oracle.ACT_SILU, oracle.ACT_GELU_TANH, oracle.ACT_GELU_ERF):
        d = fn(x, None, None, act) - fn(-x, None, None, act)
        if not np.allclose(d, x, rtol=0, atol=1e-12):
            return False
    return True


def pin_matches_torch(fn) -> bool:
    x = np.random.default_rng(0).normal(0, 3, (4, 50))
    for act in ACTS:
        if not np.allclose(fn(x, None, None, act), torch_act(x, act), rtol=1e-13, atol=1e-15):
            return False
    return True


def pin_bias_and_residual_exact(fn) -> bool:
    """Integer C, bias and residual: relu(C + bias[col]) + residual is exact."""
    rng = np.random.default_rng(1)
    C = rng.integers(-50, 50, (3, 5)).astype(np.float64)
    bias = rng.integers(-10, 10, 5).astype(np.float32)
    res = rng.integers(-5, 5, (3, 5)).astype(np.float32)
    got = fn(C, bias, res, oracle.ACT_RELU)
    expect = np.maximum(C + bias[None, :], 0.0) + res
    return np.array_equal(got, expect)


def pin_residual_dtypes(fn) -> bool:
    """bf16 / fp16 residual patterns widen exactly (same values as fp32)."""
    C = np.zeros((2, 3))
    r32 = np.array([[1.5, -2.25, 0.125], [3.0, -0.5, 7.0]], dtype=np.float32)
    a = fn(C, None, r32, oracle.ACT_NONE)
    b = fn(C, None, torch.tensor(r32).to(torch.bfloat16), oracle.ACT_NONE)
    h = fn(C, None, torch.tensor(r32).to(torch.float16), oracle.ACT_NONE)
    return np.array_equal(a, r32.astype(np.float64)) and np.array_equal(a, b) and np.array_equal(a, h)


PINS = [pin_special_values, pin_odd_part, pin_matches_torch, pin_bias_and_residual_exact, pin_residual_dtypes]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_epilogue_oracle_passes_pin(pin):
    assert pin(real_epilogue)


def _mutant_bias_per_row(C, bias, residual, act):
    C = np.array(C, dtype=np.float64)
    if bias is not None:
        n = min(C.shape[0], len(bias))
        C[:n] += np.asarray(bias, dtype=np.float64)[:n, None]
    return oracle.epilogue(C, None, residual, act)


def _mutant_residual_first(C, bias, residual, act):
    C = np.array(C, dtype=np.float64)
    if residual is not None:
        r = residual.float().numpy() if hasattr(residual, "float") else np.asarray(residual, dtype=np.float64)
        C = C + r
    return oracle.epilogue(C, bias, None, act)


def _mutant_swap_activation(C, bias, residual, act):
    other = {oracle.ACT_SILU: oracle.ACT_GELU_ERF, oracle.ACT_GELU_ERF: oracle.ACT_SILU,
             oracle.ACT_GELU_TANH: oracle.ACT_GELU_ERF, oracle.ACT_RELU: oracle.ACT_NONE,
             oracle.ACT_NONE: oracle.ACT_RELU}[act]
    return oracle.epilogue(C, bias, residual, other)


MUTANTS = [_mutant_bias_per_row, _mutant_residual_first, _mutant_swap_activation]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_planted_epilogue_mistakes_fail(mutant):
    failed = []
    for p in PINS:
        try:
            ok = p(mutant)
        except Exception:
            ok = False
        if not ok:
            failed.append(p.__name__)
    assert failed


@pytest.mark.parametrize("act", ACTS)
def test_activation_slopes_within_parity_rule(act):
    """The slope constants of oracle.parity bound the oracle's own activations."""
    x = np.linspace(-12, 12, 48001)
    y = np.array([oracle.activation(v, act) for v in x])
    slope = np.max(np.abs(np.diff(y) / np.diff(x)))
    assert slope <= parity.ACT_SLOPE[act]
    # and |act(x)| <= |x|, which the rounding term of the rule uses
    assert np.all(np.abs(y) <= np.abs(x) + 1e-15)


def test_epilogue_rule_accepts_fp32_rounding_rejects_errors():
    rng = np.random.default_rng(3)
    C = rng.normal(0, 4, (6, 40))
    S = np.abs(C) * 3 + 1.0
    bias = rng.normal(0, 1, 40).astype(np.float32)
    res = rng.normal(0, 2, (6, 40)).astype(np.float32)
    for act in ACTS:
        ref = oracle.epilogue(C, bias, res, act)
        pre = C + bias[None, :].astype(np.float64)
        got = ref.astype(np.float32).astype(np.float64)
        assert parity.check_epilogue(got, ref, pre, S, np.abs(res), "f32", act)["ok"]
        gb = torch.tensor(ref).to(torch.bfloat16).double().numpy()
        assert parity.check_epilogue(gb, ref, pre, S, np.abs(res), "bf16", act)["ok"]
        bad = got.copy()
        bad[2, 7] += 2.0 ** -8 * S[2, 7] + 1.0
        assert not parity.check_epilogue(bad, ref, pre, S, np.abs(res), "f32", act)["ok"]
