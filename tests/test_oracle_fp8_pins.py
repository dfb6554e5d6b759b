"""Pins of the oracle's 8-bit float path (E4M3 / E5M2 inputs) against things
other than itself (no GPU needed).

* the two decoders, on all 256 patterns each, against PyTorch's float8
  conversions and against the specification's table of special values
  (tests/golden/fp8_values.txt);
* the 8-bit GEMM against an exact-rational brute force on tiny shapes, whose
  operand values come from PyTorch's decoder, not the oracle's;
* every E4M3 / E5M2 value is exact in bf16, so the 8-bit GEMM must equal the
  (separately pinned) 16-bit GEMM on the same values bit for bit, which
  catches a transposed operand, a shifted index or a dropped term;
* the dequantisation scales against a diagonal-matrix product.
``test_planted_mistakes_fail`` checks that these pins catch planted mistakes.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_blackwell_sm_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KINDS = {"e4m3": (oracle.IN_E4M3, torch.float8_e4m3fn), "e5m2": (oracle.IN_E5M2, torch.float8_e5m2)}


def torch_decode(bits: np.ndarray, tdt) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(tdt)
    return t.to(torch.float64).numpy()


def golden_rows():
    out = []
    for line in open(os.path.join(GOLDEN, "fp8_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, bits, value = (f.strip() for f in line.split("|"))
        out.append((kind, int(bits, 16), value))
    return out


def parse_value(v: str) -> float:
    if v in ("inf", "-inf", "nan"):
        return float(v)
    return float(Fraction(v))


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_decoder_matches_torch_on_every_pattern(name):
    kind, tdt = KINDS[name]
    ref = torch_decode(np.arange(256), tdt)
    got = np.array([oracle.widen8(b, kind) for b in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    # sign symmetry: flipping bit 7 negates every non-NaN value
    assert (got[0x80:][~nan[0x80:]] == -got[:0x80][~nan[0x80:]]).all()


def test_decoder_matches_the_specification_table():
    rows = golden_rows()
    assert len(rows) >= 25
    for name, bits, value in rows:
        got = oracle.widen8(bits, KINDS[name][0])
        want = parse_value(value)
        if np.isnan(want):
            assert np.isnan(got), (name, hex(bits))
        else:
            assert got == want, (name, hex(bits), got, want)


def random_fp8(M, N, K, name, seed):
    a, b = inputs.make_operands(M, N, K, name, ("normal", 1.0), ("uniform",), seed=seed)
    return a, b


def exact(a, b):
    A = [[Fraction(float(v)) for v in row] for row in a.to(torch.float64).numpy()]
    B = [[Fraction(float(v)) for v in row] for row in b.to(torch.float64).numpy()]
    C = [[sum((x * y for x, y in zip(ra, rb)), Fraction(0)) for rb in B] for ra in A]
    S = [[sum((abs(x * y) for x, y in zip(ra, rb)), Fraction(0)) for rb in B] for ra in A]
    return C, S


def pin_bruteforce(fn) -> bool:
    for name in KINDS:
        for i, (M, N, K) in enumerate([(1, 1, 1), (2, 3, 5), (3, 2, 7), (5, 7, 3), (4, 4, 16), (2, 9, 33)]):
            a, b = random_fp8(M, N, K, name, seed=10 + i)
            C, S = fn(a, b)
            Ce, Se = exact(a, b)
            for r in range(M):
                for c in range(N):
                    # products are exact in fp64; the sums of at most 33 of them round at most slightly
                    if abs(Fraction(C[r, c]) - Ce[r][c]) > Se[r][c] * Fraction(1, 2 ** 45):
                        return False
                    if abs(Fraction(S[r, c]) - Se[r][c]) > Se[r][c] * Fraction(1, 2 ** 45):
                        return False
    return True


def pin_equals_bf16_path(fn) -> bool:
    for name in KINDS:
        for i, (M, N, K) in enumerate([(7, 13, 64), (33, 5, 48), (16, 16, 160)]):
            a, b = random_fp8(M, N, K, name, seed=40 + i)
            C, S = fn(a, b)
            C16, S16 = oracle.gemm(a.to(torch.bfloat16), b.to(torch.bfloat16))
            if not (np.array_equal(C, C16) and np.array_equal(S, S16)):
                return False
    return True


def pin_rows(fn) -> bool:
    a, b = random_fp8(40, 24, 96, "e4m3", seed=7)
    C, _ = fn(a, b)
    rows = [0, 5, 39, 17]
    Cr, _ = oracle.gemm_rows(a, b, rows)
    return np.array_equal(Cr, C[rows])


def test_bruteforce():
    assert pin_bruteforce(oracle.gemm)


def test_equals_the_16bit_gemm_on_the_same_values():
    assert pin_equals_bf16_path(oracle.gemm)


def test_rows_agree_with_the_full_product():
    assert pin_rows(oracle.gemm)


def test_special_values_propagate():
    a = torch.tensor([[1.0, 2.0], [1.0, 1.0]]).to(torch.float8_e5m2)
    b = torch.tensor([[1.0, 1.0]]).to(torch.float8_e5m2)
    bits = a.view(torch.uint8).clone()
    bits[0, 1] = 0x7C        # +inf
    bits[1, 0] = 0x7D        # NaN
    C, _ = oracle.gemm(bits.view(torch.float8_e5m2), b)
    assert C[0, 0] == np.inf and np.isnan(C[1, 0])
    a4 = torch.tensor([[1.0, 2.0]]).to(torch.float8_e4m3fn)
    bits4 = a4.view(torch.uint8).clone()
    bits4[0, 0] = 0x7F       # NaN (E4M3 has no infinity)
    C4, _ = oracle.gemm(bits4.view(torch.float8_e4m3fn), a4)
    assert np.isnan(C4[0, 0])


def test_extremes_and_subnormals():
    # 448 * 448 (E4M3 max) and 2^-9 * 2^-9 (smallest subnormal) are exact
    a = torch.tensor([[448.0, 2.0 ** -9]]).to(torch.float8_e4m3fn)
    C, S = oracle.gemm(a, a)
    assert C[0, 0] == 448.0 ** 2 + 2.0 ** -18 and S[0, 0] == C[0, 0]
    b = torch.tensor([[57344.0, -(2.0 ** -16)]]).to(torch.float8_e5m2)
    C, _ = oracle.gemm(b, b)
    assert C[0, 0] == 57344.0 ** 2 + 2.0 ** -32


def test_scale_is_a_diagonal_product():
    rng = np.random.default_rng(3)
    C = rng.standard_normal((6, 5))
    sa = rng.uniform(0.5, 2.0, 6).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, 5).astype(np.float32)
    got = oracle.scale(C, sa, sb)
    want = np.diag(sa.astype(np.float64)) @ C @ np.diag(sb.astype(np.float64))
    assert np.allclose(got, want, rtol=1e-15, atol=0)
    assert np.array_equal(oracle.scale(C, None, None), C)
    assert np.array_equal(oracle.scale(C, np.ones(6), None), C)
    # the epilogue applies the scales before the bias
    bias = np.arange(5, dtype=np.float32)
    e = oracle.epilogue(C, bias=bias, scale_a=sa, scale_b=sb)
    assert np.allclose(e, want + bias, rtol=1e-15, atol=1e-15)
    with pytest.raises(ValueError):
        oracle.scale(C, sa[:5], None)


def test_rejects_bad_arguments():
    a = torch.zeros(2, 4, dtype=torch.float8_e4m3fn)
    b = torch.zeros(3, 5, dtype=torch.float8_e4m3fn)
    with pytest.raises(ValueError):
        oracle.gemm(a, b)
    with pytest.raises(ValueError):
        oracle.gemm_rows(a, a, [2])
    with pytest.raises(TypeError):
        oracle.gemm(np.zeros((2, 4), np.float32), np.zeros((2, 4), np.float32), oracle.IN_E4M3)


# ----------------------------------------------------------------------------
# planted mistakes (on the CPU, around the real oracle) must fail a pin

def _mutants():
    def transposed_b(a, b):
        C, S = oracle.gemm(a, b)
        return C.T.copy() if C.shape[0] == C.shape[1] else C[::-1].copy(), S

    def dropped_last_k(a, b):
        return oracle.gemm(a[:, :-1].contiguous(), b[:, :-1].contiguous()) if a.shape[1] > 1 else \
            (np.zeros((a.shape[0], b.shape[0])), np.zeros((a.shape[0], b.shape[0])))

    def wrong_format(a, b):
        kind = oracle.IN_E5M2 if a.dtype == torch.float8_e4m3fn else oracle.IN_E4M3
        return oracle.gemm(a, b, kind)

    def e4m3_bias_off_by_one(a, b):
        C, S = oracle.gemm(a, b)
        return (C * 2.0, S * 2.0) if a.dtype == torch.float8_e4m3fn else (C, S)

    def sign_lost(a, b):
        C, S = oracle.gemm(a, b)
        return S.copy(), S

    def shifted_row(a, b):
        C, S = oracle.gemm(a, b)
        return np.roll(C, 1, axis=0), np.roll(S, 1, axis=0)

    return [transposed_b, dropped_last_k, wrong_format, e4m3_bias_off_by_one, sign_lost, shifted_row]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_planted_mistakes_fail(mutant):
    assert not (pin_bruteforce(mutant) and pin_equals_bf16_path(mutant) and pin_rows(mutant))
