"""Roofline arithmetic for the dense GEMM and the decode GEMV.

The model is the one the reading notes of "Modern GPU Programming for MLSys"
state in section "Roofline：找到天花板": attainable FLOP/s is bounded by
min(peak compute, bandwidth x arithmetic intensity), where arithmetic
intensity is FLOPs per byte moved to or from HBM, and the ridge point is
peak / bandwidth.  FLOPs are the 2*M*N*K multiply-adds of the product; bytes are
the algorithmic minimum -- each operand read once, the result written once.
"""
from __future__ import annotations

IN_BYTES = {"f16": 2, "bf16": 2}
OUT_BYTES = {"f32": 4, "bf16": 2, "f16": 2}


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, in_bytes: int = 2, out_bytes: int = 2) -> int:
    return in_bytes * (M * K + N * K) + out_bytes * M * N


def arithmetic_intensity(M: int, N: int, K: int, in_bytes: int = 2, out_bytes: int = 2) -> float:
    return gemm_flops(M, N, K) / gemm_bytes(M, N, K, in_bytes, out_bytes)


def ridge_point(peak_flops: float, bandwidth: float) -> float:
    return peak_flops / bandwidth


def attainable(ai: float, peak_flops: float, bandwidth: float) -> float:
    return min(peak_flops, bandwidth * ai)


def bound_of(ai: float, peak_flops: float, bandwidth: float) -> str:
    return "tensor" if ai >= ridge_point(peak_flops, bandwidth) else "hbm"
