"""Acceptance rule for comparing a GPU result with the oracle -- TEST INFRASTRUCTURE.

Per element, with ``ref`` and ``S = sum_k |a_ik b_jk|`` from the oracle (fp64):

  * fp32 output:  |c - ref| <= 2^-10 * S
  * bf16 output:  |c - ref| <= 2^-10 * S + half_ulp_bf16(|ref|)
  * any NaN / Inf in c fails (the inputs are finite by construction).

``2^-10 * S`` covers an fp32 accumulation of fp16/bf16 products in any order
(the Tensor Core's internal order is unspecified), with a wide margin: a
sequential fp32 sum errs by at most about K * 2^-24 * S.  ``half_ulp_bf16`` is
the last rounding of the fp32 accumulator to bf16 (round to nearest even):
for |ref| > 0 with |ref| = m * 2^e, 0.5 <= m < 1 (frexp), bf16's 8-bit
significand gives ulp 2^(e-8) and half an ulp 2^(e-9); for ref == 0 it is 0,
so an all-zero row (S == 0) must come back as exact zeros.
"""
from __future__ import annotations

import numpy as np

TOL_REL = 2.0 ** -10


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(ref)
    h = np.ldexp(np.ones_like(ref), e.astype(np.int64) - 9)
    return np.where(ref > 0, h, 0.0)


def bound(ref: np.ndarray, S: np.ndarray, out_dtype: str) -> np.ndarray:
    b = TOL_REL * np.asarray(S, dtype=np.float64)
    if out_dtype == "bf16":
        b = b + half_ulp_bf16(ref)
    elif out_dtype != "f32":
        raise ValueError(out_dtype)
    return b


def check(c, ref: np.ndarray, S: np.ndarray, out_dtype: str) -> dict:
    """Compare ``c`` (anything convertible to float64) with the oracle.

    Returns a dict with ``ok`` plus diagnostics: the worst ratio
    |c-ref| / bound, the count of violations, the max / RMS of |c-ref| / S,
    and ``max_excess_rel``: the largest error beyond the output rounding
    (half a bf16 ulp of the larger of |c| and |ref|), relative to S, which
    fp32 accumulation keeps far below 2^-10.
    """
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    if c.shape != ref.shape or S.shape != ref.shape:
        raise ValueError("shape mismatch %s %s %s" % (c.shape, ref.shape, S.shape))
    finite = np.isfinite(c)
    err = np.abs(c - ref)
    b = bound(ref, S, out_dtype)
    bad = ~finite | (err > b)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(b > 0, err / b, np.where(err > 0, np.inf, 0.0))
        rel = np.where(S > 0, err / S, np.where(err > 0, np.inf, 0.0))
    # the error left after the output rounding is allowed for: with fp32
    # accumulation it is tiny, so a large value means a lost K block or row
    allow = half_ulp_bf16(np.maximum(np.abs(ref), np.abs(np.where(finite, c, 0.0)))) if out_dtype == "bf16" else 0.0
    excess = np.maximum(err - allow, 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        exc_rel = np.where(S > 0, excess / S, np.where(excess > 0, np.inf, 0.0))
    n = max(1, rel.size)
    out = {
        "ok": bool(not bad.any()),
        "n": int(c.size),
        "violations": int(bad.sum()),
        "nonfinite": int((~finite).sum()),
        "worst_ratio": float(np.max(ratio)) if ratio.size else 0.0,
        "max_rel": float(np.max(rel)) if rel.size else 0.0,
        "rms_rel": float(np.sqrt(np.sum(np.where(np.isfinite(rel), rel, 0.0) ** 2) / n)),
        "max_excess_rel": float(np.max(np.where(finite, exc_rel, np.inf))) if exc_rel.size else 0.0,
    }
    if bad.any():
        idx = np.argwhere(bad)[0]
        out["first_bad"] = {"index": [int(i) for i in idx], "c": float(c[tuple(idx)]),
                            "ref": float(ref[tuple(idx)]), "S": float(S[tuple(idx)])}
    return out


# Largest slope of each activation (0 none, 1 relu, 2 silu, 3 gelu-tanh,
# 4 gelu-erf): silu' peaks at 1.0998 (x ~ 2.40), both gelu forms at 1.1289
# (x ~ 1.41 for erf, ~1.44 for tanh); pinned numerically by the oracle tests.
ACT_SLOPE = {0: 1.0, 1: 1.0, 2: 1.1, 3: 1.13, 4: 1.13}
EPI_REL = 2.0 ** -17


def epilogue_bound(ref_epi, pre, S, residual_abs, out_dtype: str, act: int) -> np.ndarray:
    """Per-element bound for C = act(acc + bias) + residual.

    An accumulator error e (|e| <= 2^-10 S, the GEMM rule) moves act(.) by at
    most slope * e; the fp32 additions of bias and residual and the fp32
    activation (the kernels' SiLU and tanh-form GeLU go through the hardware's
    approximate exp2 and reciprocal, the erf form through CUDA's erff) add at most
    2^-17 (|acc + bias| + |residual|), since |act(x)| <= |x| for every
    activation here; bf16 output adds half an ulp of the final value."""
    b = ACT_SLOPE[act] * TOL_REL * np.asarray(S, dtype=np.float64)
    b = b + EPI_REL * (np.abs(np.asarray(pre, dtype=np.float64)) + np.asarray(residual_abs, dtype=np.float64))
    if out_dtype == "bf16":
        b = b + half_ulp_bf16(ref_epi)
    return b


def check_epilogue(c, ref_epi, pre, S, residual_abs, out_dtype: str, act: int) -> dict:
    c = np.asarray(c, dtype=np.float64)
    ref_epi = np.asarray(ref_epi, dtype=np.float64)
    finite = np.isfinite(c)
    err = np.abs(c - ref_epi)
    b = epilogue_bound(np.maximum(np.abs(ref_epi), np.abs(np.where(finite, c, 0.0))), pre, S, residual_abs,
                       out_dtype, act)
    bad = ~finite | (err > b)
    out = {"ok": bool(not bad.any()), "violations": int(bad.sum()),
           "worst_ratio": float(np.max(np.where(b > 0, err / np.where(b > 0, b, 1.0), np.where(err > 0, np.inf, 0.0))))}
    if bad.any():
        idx = np.argwhere(bad)[0]
        out["first_bad"] = {"index": [int(i) for i in idx], "c": float(c[tuple(idx)]),
                            "ref": float(ref_epi[tuple(idx)]), "bound": float(b[tuple(idx)])}
    return out
