"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each pin is written so that a plausible mistake in the oracle -- a dropped
k-term, a wrong sign, a transposed operand or result, a shifted index, a bad
16-bit decoder -- fails at least one of them; ``test_planted_mistakes_fail``
plants those mistakes around the real oracle and checks exactly that.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import inputs, roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F16, BF16 = oracle.IN_F16, oracle.IN_BF16


# ----------------------------------------------------------------------------
# independent decoders (numpy's IEEE conversions), used only by the pins

def np_decode(bits: np.ndarray, kind: int) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if kind == F16:
        return bits.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def exact_gemm(a_bits, b_bits, kind):
    """Exact rationals C and S by brute force (fractions.Fraction)."""
    A = [[Fraction(float(v)) for v in row] for row in np_decode(a_bits, kind)]
    B = [[Fraction(float(v)) for v in row] for row in np_decode(b_bits, kind)]
    C = [[sum((x * y for x, y in zip(ra, rb)), Fraction(0)) for rb in B] for ra in A]
    S = [[sum((abs(x * y) for x, y in zip(ra, rb)), Fraction(0)) for rb in B] for ra in A]
    return C, S


def real_oracle(a_bits, b_bits, kind):
    return oracle.gemm(a_bits, b_bits, kind)


# ----------------------------------------------------------------------------
# pins as reusable checks on an oracle-like function fn(a_bits, b_bits, kind)

def pin_bruteforce(fn, seed=0) -> bool:
    rng = np.random.default_rng(seed)
    for kind in (F16, BF16):
        for (M, N, K) in [(1, 1, 1), (2, 3, 5), (3, 2, 7), (5, 7, 3), (7, 5, 16), (16, 3, 2), (2, 16, 16)]:
            dt = torch.float16 if kind == F16 else torch.bfloat16
            a = torch.tensor(rng.uniform(-1, 1, (M, K)), dtype=torch.float32).to(dt)
            b = torch.tensor(rng.standard_normal((N, K)) * 3.0, dtype=torch.float32).to(dt)
            ab, bb = to_bits(a), to_bits(b)
            C, S = fn(ab, bb, kind)
            Ce, Se = exact_gemm(ab, bb, kind)
            if C.shape != (M, N):
                return False
            for i in range(M):
                for j in range(N):
                    tol = float(Se[i][j]) * 2.0 ** -50
                    if abs(Fraction(float(C[i, j])) - Ce[i][j]) > Fraction(tol):
                        return False
                    if abs(Fraction(float(S[i, j])) - Se[i][j]) > Fraction(tol):
                        return False
    return True


def pin_identity(fn) -> bool:
    """A = I (M = K): C = B^T exactly; B = I (N = K): C = A exactly."""
    rng = np.random.default_rng(1)
    K, N = 16, 9
    for kind in (F16, BF16):
        dt = torch.float16 if kind == F16 else torch.bfloat16
        eye = to_bits(torch.eye(K, dtype=dt))
        b = to_bits(torch.tensor(rng.uniform(-4, 4, (N, K)), dtype=torch.float32).to(dt))
        C, _ = fn(eye, b, kind)
        if C.shape != (K, N) or not np.array_equal(C, np_decode(b, kind).T):
            return False
        a = to_bits(torch.tensor(rng.uniform(-4, 4, (N, K)), dtype=torch.float32).to(dt))
        C2, _ = fn(a, eye, kind)
        if C2.shape != (N, K) or not np.array_equal(C2, np_decode(a, kind)):
            return False
    return True


def pin_permutation(fn) -> bool:
    """A = P (a permutation matrix, P[i, p(i)] = 1): C[i, j] = b[j, p(i)].
    B is square (N = K) and not symmetric, so reading B untransposed fails."""
    rng = np.random.default_rng(2)
    K, N = 12, 12
    p = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[np.arange(K), p] = 1.0
    for kind in (F16, BF16):
        dt = torch.float16 if kind == F16 else torch.bfloat16
        Pb = to_bits(torch.tensor(P).to(dt))
        b = to_bits(torch.tensor(rng.uniform(-8, 8, (N, K)), dtype=torch.float32).to(dt))
        C, _ = fn(Pb, b, kind)
        if C.shape != (K, N):
            return False
        expect = np_decode(b, kind)[:, p].T
        if not np.array_equal(C, expect):
            return False
    return True


def pin_rank1(fn) -> bool:
    """a[i,k] = u_i w_k, b[j,k] = v_j z_k with small dyadic values, so every
    product is exact: C[i,j] = u_i v_j sum_k w_k z_k exactly."""
    rng = np.random.default_rng(3)
    M, N, K = 6, 5, 24
    u = rng.integers(-3, 4, M) * 0.5
    v = rng.integers(-3, 4, N) * 0.25
    w = rng.integers(-4, 5, K).astype(np.float64)
    z = rng.integers(-2, 3, K) * 2.0
    for kind in (F16, BF16):
        dt = torch.float16 if kind == F16 else torch.bfloat16
        a = to_bits(torch.tensor(np.outer(u, w), dtype=torch.float32).to(dt))
        b = to_bits(torch.tensor(np.outer(v, z), dtype=torch.float32).to(dt))
        C, S = fn(a, b, kind)
        expect = np.outer(u, v) * float(np.dot(w, z))
        expect_s = np.outer(np.abs(u), np.abs(v)) * float(np.dot(np.abs(w), np.abs(z)))
        if C.shape != (M, N) or not np.array_equal(C, expect) or not np.array_equal(S, expect_s):
            return False
    return True


def pin_transpose_symmetry(fn) -> bool:
    """oracle(B, A) == oracle(A, B)^T exactly (products commute, same k order)."""
    a, b = inputs.make_operands(9, 13, 40, "bf16", ("normal", 1.0), ("uniform",), seed=5)
    ab, bb = to_bits(a), to_bits(b)
    C1, S1 = fn(ab, bb, BF16)
    C2, S2 = fn(bb, ab, BF16)
    return C1.shape == (9, 13) and np.array_equal(C1, C2.T) and np.array_equal(S1, S2.T)


def pin_additivity(fn) -> bool:
    """oracle(A1 + A2, B) == oracle(A1, B) + oracle(A2, B) within 2^-40 S, with
    A1 + A2 exactly representable (small integers)."""
    rng = np.random.default_rng(6)
    M, N, K = 5, 6, 64
    A1 = rng.integers(-8, 9, (M, K)).astype(np.float32)
    A2 = rng.integers(-8, 9, (M, K)).astype(np.float32)
    Bf = rng.uniform(-1, 1, (N, K)).astype(np.float32)
    dt = torch.float16
    b = to_bits(torch.tensor(Bf).to(dt))
    C12, S12 = fn(to_bits(torch.tensor(A1 + A2).to(dt)), b, F16)
    C1, S1 = fn(to_bits(torch.tensor(A1).to(dt)), b, F16)
    C2, S2 = fn(to_bits(torch.tensor(A2).to(dt)), b, F16)
    tol = 2.0 ** -40 * (S1 + S2)
    return C12.shape == (M, N) and bool(np.all(np.abs(C12 - (C1 + C2)) <= tol))


PINS = [pin_bruteforce, pin_identity, pin_permutation, pin_rank1,
        pin_transpose_symmetry, pin_additivity]


# ----------------------------------------------------------------------------
# the tests

@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_passes_pin(pin):
    assert pin(real_oracle)


def _mutant_drop_last_term(a, b, kind):
    return oracle.gemm(np.ascontiguousarray(a[:, :-1]), np.ascontiguousarray(b[:, :-1]), kind)


def _mutant_negate(a, b, kind):
    C, S = oracle.gemm(a, b, kind)
    return -C, S


def _mutant_swap_operands(a, b, kind):
    return oracle.gemm(b, a, kind)


def _mutant_transpose_b(a, b, kind):
    # C = A * B (B read as K x N) -- only shape-valid when B is square
    if b.shape[0] != b.shape[1]:
        return oracle.gemm(a, b, kind)
    return oracle.gemm(a, np.ascontiguousarray(b.T), kind)


def _mutant_shift_k(a, b, kind):
    # index slip: a[i, k] paired with b[j, (k + 1) % K]
    return oracle.gemm(a, np.ascontiguousarray(np.roll(b, -1, axis=1)), kind)


def _mutant_bf16_as_f16(a, b, kind):
    return oracle.gemm(a, b, F16 if kind == BF16 else BF16)


MUTANTS = [_mutant_drop_last_term, _mutant_negate, _mutant_swap_operands,
           _mutant_transpose_b, _mutant_shift_k, _mutant_bf16_as_f16]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_planted_mistakes_fail(mutant):
    def safe(pin):
        try:
            return pin(mutant)
        except Exception:
            return False
    failed = [p.__name__ for p in PINS if not safe(p)]
    assert failed, "a planted mistake passed every pin"


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


def _frac(s: str) -> Fraction:
    if "*" in s:
        x, y = s.split("*")
        return Fraction(x) * Fraction(y)
    return Fraction(s)


def test_decoders_match_format_definitions():
    rows = _golden_rows("half_precision_values.txt")
    assert len(rows) >= 20
    for kind_s, bits_s, val_s in rows:
        kind = F16 if kind_s == "f16" else BF16
        got = oracle.widen(int(bits_s, 16), kind)
        assert Fraction(got) == _frac(val_s), (kind_s, bits_s, got, val_s)


@pytest.mark.parametrize("kind", [F16, BF16], ids=["f16", "bf16"])
def test_decoder_exhaustive_against_numpy(kind):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = np_decode(bits, kind)
    got = np.array([oracle.widen(int(b), kind) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the sign of zero too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_rows_subset_equals_full():
    a, b = inputs.make_operands(37, 29, 72, "f16", ("uniform",), ("uniform",), seed=7)
    C, S = oracle.gemm(a, b)
    rows = [0, 36, 5, 17, 5]
    Cr, Sr = oracle.gemm_rows(a, b, rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])


def test_thread_count_does_not_change_bits():
    a, b = inputs.make_operands(33, 20, 200, "bf16", ("normal", 0.02), ("normal", 0.02), seed=8)
    C1, S1 = oracle.gemm(a, b, nthreads=1)
    C4, S4 = oracle.gemm(a, b, nthreads=4)
    assert np.array_equal(C1, C4) and np.array_equal(S1, S4)


def test_zero_row_is_exact_zero():
    a, b = inputs.make_operands(4, 5, 16, "bf16", ("uniform",), ("uniform",), seed=9)
    a[2].zero_()
    C, S = oracle.gemm(a, b)
    assert np.all(C[2] == 0.0) and np.all(S[2] == 0.0)


def test_integer_inputs_exact():
    a, b = inputs.integer_operands(20, 24, 300, "bf16", seed=10)
    C, _ = oracle.gemm(a, b)
    ref = a.to(torch.float64) @ b.to(torch.float64).T   # integers: exact in any order
    assert np.array_equal(C, ref.numpy())


def test_roofline_worked_examples():
    for row in _golden_rows("roofline_worked_examples.txt"):
        kind, name, M, N, K, ib, ob, peak, bw, printed, slack, bound = row
        peak, bw, printed, slack = float(peak), float(bw), float(printed), float(slack)
        if kind == "ridge":
            assert roofline.ridge_point(peak, bw) == printed, name
            continue
        ai = roofline.arithmetic_intensity(int(M), int(N), int(K), int(ib), int(ob))
        assert abs(ai - printed) <= slack * printed, (name, ai)
        assert roofline.bound_of(ai, peak, bw) == bound, name
    # the two closed forms behind the printed numbers
    assert roofline.arithmetic_intensity(4096, 4096, 4096, 2, 2) == pytest.approx(4096 / 3)
    assert roofline.arithmetic_intensity(4096, 4096, 4096, 2, 4) == pytest.approx(1024.0)


# ----------------------------------------------------------------------------
# the acceptance rule itself

def test_half_ulp_bf16_values():
    got = parity.half_ulp_bf16(np.array([1.0, 1.5, 0.75, -3.0, 0.0, 2.0 ** -20]))
    # bf16 keeps 8 significand bits: ulp(1) = 2^-7, so half an ulp at 1 is 2^-8
    assert list(got) == [2.0 ** -8, 2.0 ** -8, 2.0 ** -9, 2.0 ** -7, 0.0, 2.0 ** -28]


def test_parity_rule_accepts_rounding_and_rejects_errors():
    a, b = inputs.make_operands(16, 24, 256, "bf16", ("uniform",), ("uniform",), seed=11)
    C, S = oracle.gemm(a, b)
    c32 = torch.tensor(C).to(torch.float32)
    assert parity.check(c32.numpy(), C, S, "f32")["ok"]
    cb = c32.to(torch.bfloat16).to(torch.float64).numpy()        # RN to bf16
    assert parity.check(cb, C, S, "bf16")["ok"]
    bad = c32.numpy().astype(np.float64).copy()
    bad[3, 5] += 2.0 ** -9 * S[3, 5]
    r = parity.check(bad, C, S, "f32")
    assert not r["ok"] and r["violations"] == 1 and r["first_bad"]["index"] == [3, 5]
    nan = c32.numpy().copy()
    nan[0, 0] = np.nan
    assert not parity.check(nan, C, S, "f32")["ok"]


def test_parity_rule_zero_sum_must_be_exact_zero():
    ref = np.zeros((2, 2))
    S = np.zeros((2, 2))
    assert parity.check(np.zeros((2, 2)), ref, S, "bf16")["ok"]
    assert parity.check(-np.zeros((2, 2)), ref, S, "f32")["ok"]
    c = np.zeros((2, 2))
    c[1, 1] = 1e-30
    assert not parity.check(c, ref, S, "f32")["ok"]


# ----------------------------------------------------------------------------
# the seeded input recipe

def test_inputs_are_reproducible_and_drawn_a_then_b():
    a1, b1 = inputs.make_operands(8, 6, 32, "f16", ("uniform",), ("uniform",), seed=3)
    a2, b2 = inputs.make_operands(8, 6, 32, "f16", ("uniform",), ("uniform",), seed=3)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    g = torch.Generator().manual_seed(3)
    ra = (torch.rand(8, 32, generator=g) * 2 - 1).to(torch.float16)
    rb = (torch.rand(6, 32, generator=g) * 2 - 1).to(torch.float16)
    assert torch.equal(a1, ra) and torch.equal(b1, rb)
    assert float(a1.abs().max()) <= 1.0


def test_workload_table_shapes():
    w = inputs.WORKLOADS
    assert (w["large_8192_bf16_bf16"].M, w["large_8192_bf16_bf16"].N, w["large_8192_bf16_bf16"].K) == (8192,) * 3
    assert w["single_tile_128x128x64_f16_f32"].seed == 0
    assert w["gemv_m1_n4096_k4096_bf16"].M == 1
    assert w["square_4096_f16_f32"].algorithmic_bytes == 2 * 2 * 4096 * 4096 + 4 * 4096 * 4096
    assert w["fp8_8192_e4m3_bf16"].algorithmic_bytes == 2 * 8192 * 8192 + 2 * 8192 * 8192


def test_parity_diagnostic_flags_a_lost_k_block():
    a, b = inputs.make_operands(8, 16, 512, "bf16", ("uniform",), ("uniform",), seed=12)
    C, S = oracle.gemm(a, b)
    good = torch.tensor(C).to(torch.bfloat16).to(torch.float64).numpy()
    assert parity.check(good, C, S, "bf16")["max_excess_rel"] < 2.0 ** -16
    # the same product with the last 64-wide K block left out
    Cd, _ = oracle.gemm(a[:, :448].contiguous(), b[:, :448].contiguous())
    lost = torch.tensor(Cd).to(torch.bfloat16).to(torch.float64).numpy()
    assert parity.check(lost, C, S, "bf16")["max_excess_rel"] > 2.0 ** -12
