"""Pins of the oracle's MX block-scaled product (``oracle.gemm_mx``: 8-bit
float operands, one UE8M0 scale per 32 consecutive K elements of every row of
A and of B) against things other than itself (no GPU needed):

* the UE8M0 decoder on all 256 bytes against PyTorch's float8_e8m0fnu;
* unit scales (byte 127) reduce it to the separately pinned 8-bit GEMM;
* per-row / per-column constant scales reduce it to that GEMM times the
  (pinned) diagonal dequantisation scales;
* varying scales equal the sum over 32-wide K slices of scaled slice GEMMs;
* an exact-rational brute force on tiny shapes with PyTorch's decoders;
* the tiled scale layout of the input generator is checked index by index.
``test_planted_mistakes_fail`` checks that these pins catch planted mistakes.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_blackwell_sm_gb300 import inputs


def ue8m0_torch(s) -> np.ndarray:
    t = torch.as_tensor(np.asarray(s, dtype=np.uint8)).contiguous()
    return t.view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def test_ue8m0_decoder_matches_torch():
    ref = ue8m0_torch(np.arange(256))
    got = np.array([oracle.ue8m0(e) for e in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert (got[:255] == ref[:255]).all()
    assert oracle.ue8m0(127) == 1.0 and oracle.ue8m0(128) == 2.0 and oracle.ue8m0(0) == 2.0 ** -127


def pin_unit_scales(fn) -> bool:
    for i, fmt in enumerate(("e4m3", "e5m2")):
        M, N, K = 9, 12, 96
        a, b, _, _ = inputs.mx_operands(M, N, K, fmt, seed=3 + i)
        one_a = torch.full((M, 3), 127, dtype=torch.uint8)
        one_b = torch.full((N, 3), 127, dtype=torch.uint8)
        C, S = fn(a, b, one_a, one_b)
        C0, S0 = oracle.gemm(a, b)
        if not (np.array_equal(C, C0) and np.array_equal(S, S0)):
            return False
    return True


def pin_row_col_constant(fn) -> bool:
    M, N, K = 17, 10, 160
    a, b, _, _ = inputs.mx_operands(M, N, K, "e4m3", seed=8)
    g = torch.Generator().manual_seed(1)
    ea = torch.randint(118, 137, (M, 1), generator=g).to(torch.uint8)
    eb = torch.randint(118, 137, (N, 1), generator=g).to(torch.uint8)
    C, S = fn(a, b, ea.expand(M, 5).contiguous(), eb.expand(N, 5).contiguous())
    sa = 2.0 ** (ea.double().flatten() - 127)
    sb = 2.0 ** (eb.double().flatten() - 127)
    C0, S0 = oracle.gemm(a, b)
    return np.array_equal(C, oracle.scale(C0, sa.float(), sb.float())) and \
        np.array_equal(S, oracle.scale(S0, sa.float(), sb.float()))


def pin_block_slices(fn) -> bool:
    for i, (M, N, K) in enumerate([(6, 7, 96), (5, 4, 144), (3, 9, 32)]):
        a, b, sa, sb = inputs.mx_operands(M, N, K, "e5m2" if i % 2 else "e4m3", seed=20 + i)
        C, S = fn(a, b, sa, sb)
        want = np.zeros((M, N))
        wantS = np.zeros((M, N))
        for kb in range((K + 31) // 32):
            lo, hi = 32 * kb, min(K, 32 * kb + 32)
            Cb, Sb = oracle.gemm(a[:, lo:hi].contiguous(), b[:, lo:hi].contiguous())
            xa = torch.tensor(ue8m0_torch(sa[:, kb])).float()
            xb = torch.tensor(ue8m0_torch(sb[:, kb])).float()
            want += oracle.scale(Cb, xa, xb)
            wantS += oracle.scale(Sb, xa, xb)
        if not (np.allclose(C, want, rtol=0, atol=0) or
                np.all(np.abs(C - want) <= 2.0 ** -48 * wantS)):
            return False
        if not np.all(np.abs(S - wantS) <= 2.0 ** -48 * wantS):
            return False
    return True


def pin_bruteforce(fn) -> bool:
    for i, (M, N, K) in enumerate([(1, 1, 16), (2, 3, 48), (3, 2, 64), (2, 2, 80)]):
        a, b, sa, sb = inputs.mx_operands(M, N, K, "e4m3", seed=50 + i, e_lo=124, e_hi=130)
        C, S = fn(a, b, sa, sb)
        av, bv = a.to(torch.float64).numpy(), b.to(torch.float64).numpy()
        xa, xb = ue8m0_torch(sa.numpy()), ue8m0_torch(sb.numpy())
        for r in range(M):
            for c in range(N):
                terms = [Fraction(float(xa[r, k // 32])) * Fraction(float(av[r, k])) *
                         Fraction(float(xb[c, k // 32])) * Fraction(float(bv[c, k])) for k in range(K)]
                ex, exs = sum(terms, Fraction(0)), sum((abs(t) for t in terms), Fraction(0))
                if abs(Fraction(C[r, c]) - ex) > exs * Fraction(1, 2 ** 48):
                    return False
                if abs(Fraction(S[r, c]) - exs) > exs * Fraction(1, 2 ** 48):
                    return False
    return True


PINS = [pin_unit_scales, pin_row_col_constant, pin_block_slices, pin_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    assert pin(oracle.gemm_mx)


def test_rows_and_nan_scale():
    a, b, sa, sb = inputs.mx_operands(40, 12, 64, "e4m3", seed=2)
    C, S = oracle.gemm_mx(a, b, sa, sb)
    Cr, Sr = oracle.gemm_mx(a, b, sa, sb, rows=[39, 0, 7])
    assert np.array_equal(Cr, C[[39, 0, 7]]) and np.array_equal(Sr, S[[39, 0, 7]])
    sa2 = sa.clone()
    sa2[3, 1] = 255
    C2, _ = oracle.gemm_mx(a, b, sa2, sb)
    assert np.isnan(C2[3]).all() and np.array_equal(np.delete(C2, 3, 0), np.delete(C, 3, 0))


def test_rejects_bad_arguments():
    a, b, sa, sb = inputs.mx_operands(4, 4, 64, "e4m3", seed=1)
    with pytest.raises(ValueError):
        oracle.gemm_mx(a, b, sa[:, :1], sb)
    with pytest.raises(ValueError):
        oracle.gemm_mx(a.to(torch.bfloat16), b.to(torch.bfloat16), sa, sb)
    with pytest.raises(ValueError):
        oracle.gemm_mx(a, b, sa, sb, rows=[4])


def test_tiled_layout_index_by_index():
    g = torch.Generator().manual_seed(4)
    for rows, K in [(1, 32), (130, 272), (256, 128), (77, 48)]:
        s = torch.randint(0, 256, (rows, (K + 31) // 32), generator=g, dtype=torch.int32).to(torch.uint8)
        t = inputs.mx_tile_scales(s, K, pad=7)
        ncb = (K + 127) // 128
        assert t.numel() == inputs.mx_tiled_bytes(rows, K) == ((rows + 127) // 128) * ncb * 512
        seen = np.zeros(t.numel(), bool)
        for r in range(rows):
            for c in range(s.shape[1]):
                off = ((r // 128) * ncb + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
                assert int(t[off]) == int(s[r, c])
                seen[off] = True
        assert (t.numpy()[~seen] == 7).all()


# ----------------------------------------------------------------------------
# planted mistakes (on the CPU, around the real oracle) must fail a pin

def _expand(s, K, block):
    """Per-element scale values for a block size `block` (the mutants' reading)."""
    x = ue8m0_torch(np.asarray(s))
    idx = np.minimum(np.arange(K) // block, x.shape[1] - 1)
    return x[:, idx]


def _via_scaled_operands(a, b, xa, xb):
    av = a.to(torch.float64).numpy() * xa
    bv = b.to(torch.float64).numpy() * xb
    return av @ bv.T, np.abs(av) @ np.abs(bv).T


def _mutants():
    def block16(a, b, sa, sb):
        K = a.shape[1]
        return _via_scaled_operands(a, b, _expand(sa, K, 16), _expand(sb, K, 16))

    def swapped_scales(a, b, sa, sb):
        if sa.shape == sb.shape:
            return oracle.gemm_mx(a, b, sb, sa)
        K = a.shape[1]
        return _via_scaled_operands(a, b, _expand(sa, K, 32), np.ones((b.shape[0], K)))

    def only_a_scaled(a, b, sa, sb):
        K = a.shape[1]
        return _via_scaled_operands(a, b, _expand(sa, K, 32), np.ones((b.shape[0], K)))

    def bias_126(a, b, sa, sb):
        C, S = oracle.gemm_mx(a, b, sa, sb)
        return C * 4.0, S * 4.0

    def last_block_unscaled(a, b, sa, sb):
        K = a.shape[1]
        xa, xb = _expand(sa, K, 32), _expand(sb, K, 32)
        xa[:, 32 * ((K - 1) // 32):] = 1.0
        return _via_scaled_operands(a, b, xa, xb)

    return [block16, swapped_scales, only_a_scaled, bias_126, last_block_unscaled]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_planted_mistakes_fail(mutant):
    assert not all(pin(mutant) for pin in PINS)


def test_the_real_oracle_agrees_with_the_mutant_harness():
    # the harness that builds the mutants is itself right when unmutated
    a, b, sa, sb = inputs.mx_operands(5, 6, 96, "e4m3", seed=9)
    C, S = oracle.gemm_mx(a, b, sa, sb)
    C2, S2 = _via_scaled_operands(a, b, _expand(sa, 96, 32), _expand(sb, 96, 32))
    assert np.allclose(C, C2, rtol=1e-12, atol=1e-12 * S.max())
