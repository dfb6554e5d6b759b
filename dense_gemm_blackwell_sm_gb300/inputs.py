"""Seeded synthetic operands for the GEMM / GEMV workloads.

This module draws random numbers and rounds them to fp16 / bf16; it holds none
of the GEMM's arithmetic.  It is the one piece the CUDA path's tests, the bench
and the CPU oracle's tests share: both sides read the very same rounded bytes.

Recipe (the pages name no RNG, so this is the plainest reading):
  * one CPU ``torch.Generator`` seeded with the workload's seed;
  * A is drawn first, then B, both in fp32, from that one generator;
  * uniform[-1, 1] is ``2 * rand - 1``; normal(0, s) is ``randn * s``;
    "normal(0,1)/sqrt(K)" is ``randn * (1/sqrt(K))``;
  * the fp32 draws are rounded to fp16 / bf16 / fp8 (E4M3, E5M2) by ``Tensor.to``
    (round to nearest even);
  * for the decode GEMV, "A" is the activation row block x (M x K) and "B" is
    the weight (N x K).
"""
from __future__ import annotations

import dataclasses
import math

import torch

F16 = "f16"
BF16 = "bf16"
F32 = "f32"
E4M3 = "e4m3"
E5M2 = "e5m2"
MXE4M3 = "mxe4m3"   # E4M3 elements with a UE8M0 scale per 32 K elements
MXE5M2 = "mxe5m2"

_TORCH = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32,
          E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2,
          MXE4M3: torch.float8_e4m3fn, MXE5M2: torch.float8_e5m2}
EIGHT_BIT = (E4M3, E5M2, MXE4M3, MXE5M2)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    in_dtype: str          # "f16" | "bf16" | "e4m3" | "e5m2" | "mxe4m3" | "mxe5m2"
    out_dtype: str         # "f32" | "bf16"
    dist_a: tuple          # ("uniform",) | ("normal", sigma) | ("normal_rsqrt_k",)
    dist_b: tuple
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        ib = 1 if self.in_dtype in EIGHT_BIT else 2
        ob = 4 if self.out_dtype == F32 else 2
        sc = ((self.M + self.N) * ((self.K + 31) // 32)) if self.in_dtype in (MXE4M3, MXE5M2) else 0
        return ib * (self.M * self.K + self.N * self.K) + ob * self.M * self.N + sc


U = ("uniform",)
N002 = ("normal", 0.02)

# The five workload families of the dense GEMM / decode GEMV, with their seeds.
WORKLOADS = {
    "single_tile_128x128x64_f16_f32": Workload("single_tile_128x128x64_f16_f32", 128, 128, 64, F16, F32, U, U, 0),
    "kloop_1024x1024x4096_bf16_bf16": Workload("kloop_1024x1024x4096_bf16_bf16", 1024, 1024, 4096, BF16, BF16,
                                               ("normal_rsqrt_k",), ("normal_rsqrt_k",), 1),
    "square_4096_f16_f32": Workload("square_4096_f16_f32", 4096, 4096, 4096, F16, F32, U, U, 2),
    "large_8192_bf16_bf16": Workload("large_8192_bf16_bf16", 8192, 8192, 8192, BF16, BF16, N002, N002, 3),
    "llm_proj_8192x14336x4096_bf16_bf16": Workload("llm_proj_8192x14336x4096_bf16_bf16", 8192, 14336, 4096,
                                                   BF16, BF16, N002, N002, 3),
    "fp8_8192_e4m3_bf16": Workload("fp8_8192_e4m3_bf16", 8192, 8192, 8192, E4M3, BF16, U, U, 5),
    "mxfp8_8192_e4m3_bf16": Workload("mxfp8_8192_e4m3_bf16", 8192, 8192, 8192, MXE4M3, BF16, U, U, 6),
    "gemv_m1_n4096_k4096_bf16": Workload("gemv_m1_n4096_k4096_bf16", 1, 4096, 4096, BF16, BF16, U, N002, 4),
    "gemv_m8_n4096_k4096_bf16": Workload("gemv_m8_n4096_k4096_bf16", 8, 4096, 4096, BF16, BF16, U, N002, 4),
    "gemv_m1_n14336_k4096_bf16": Workload("gemv_m1_n14336_k4096_bf16", 1, 14336, 4096, BF16, BF16, U, N002, 4),
    "gemv_m8_n14336_k4096_bf16": Workload("gemv_m8_n14336_k4096_bf16", 8, 14336, 4096, BF16, BF16, U, N002, 4),
}


def _draw(gen: torch.Generator, rows: int, cols: int, dist: tuple, K: int) -> torch.Tensor:
    if dist[0] == "uniform":
        return torch.rand(rows, cols, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist[0] == "normal":
        return torch.randn(rows, cols, generator=gen, dtype=torch.float32) * float(dist[1])
    if dist[0] == "normal_rsqrt_k":
        return torch.randn(rows, cols, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(K))
    if dist[0] == "int":
        lo, hi = int(dist[1]), int(dist[2])
        return torch.randint(lo, hi + 1, (rows, cols), generator=gen).to(torch.float32)
    raise ValueError("unknown distribution %r" % (dist,))


def make_operands(M: int, N: int, K: int, in_dtype: str, dist_a: tuple, dist_b: tuple, seed: int,
                  rows_a: int | None = None):
    """Seeded (A, B) as CPU fp16 / bf16 / fp8 tensors: A is M x K, B is N x K (A drawn first)."""
    gen = torch.Generator().manual_seed(int(seed))
    a = _draw(gen, M if rows_a is None else rows_a, K, dist_a, K).to(_TORCH[in_dtype])
    b = _draw(gen, N, K, dist_b, K).to(_TORCH[in_dtype])
    return a.contiguous(), b.contiguous()


def workload_operands(w: Workload):
    return make_operands(w.M, w.N, w.K, w.in_dtype, w.dist_a, w.dist_b, w.seed)


def workload_mx_scales(w: Workload):
    """Row-major UE8M0 block scales (scale_a, scale_b) of a block-scaled workload."""
    return mx_scales(w.M, w.K, w.seed + 1000), mx_scales(w.N, w.K, w.seed + 2000)


def integer_operands(M: int, N: int, K: int, in_dtype: str, seed: int, lo: int = -2, hi: int = 2):
    """Integer-valued operands in [lo, hi]: every fp32 partial sum is exact when
    K * max|a| * max|b| < 2^24, so any summation order gives the same bits."""
    return make_operands(M, N, K, in_dtype, ("int", lo, hi), ("int", lo, hi), seed)


def mx_scales(rows: int, K: int, seed: int, e_lo: int = 120, e_hi: int = 134) -> torch.Tensor:
    """Seeded UE8M0 block scales (exponent bytes uniform in [e_lo, e_hi], i.e.
    scales 2^(e_lo-127) .. 2^(e_hi-127)), row-major rows x ceil(K/32), uint8."""
    gen = torch.Generator().manual_seed(int(seed))
    return torch.randint(e_lo, e_hi + 1, (rows, (K + 31) // 32), generator=gen, dtype=torch.int32).to(torch.uint8)


def mx_operands(M: int, N: int, K: int, in_dtype: str, seed: int, dist_a: tuple = ("uniform",),
                dist_b: tuple = ("normal", 1.0), e_lo: int = 120, e_hi: int = 134):
    """(A, B, scale_a, scale_b): seeded 8-bit operands plus row-major UE8M0 block
    scales for every 32 consecutive K elements of each row."""
    a, b = make_operands(M, N, K, in_dtype, dist_a, dist_b, seed)
    return a, b, mx_scales(M, K, seed + 1000, e_lo, e_hi), mx_scales(N, K, seed + 2000, e_lo, e_hi)


def mx_tiled_bytes(rows: int, K: int) -> int:
    """Bytes of the tiled scale layout for `rows` rows: 512-byte blocks of 128 rows x 4 scales."""
    return ((rows + 127) // 128) * ((K + 127) // 128) * 512


def mx_tile_scales(s: torch.Tensor, K: int, pad: int = 127) -> torch.Tensor:
    """Row-major rows x ceil(K/32) scales rearranged (a pure permutation) into the
    tiled layout the block-scaled kernels read: 512-byte blocks, one per 128 rows
    x 4 scale columns, blocks ordered by row block then column block; inside a
    block, scale (r, c) sits at byte (r % 32) * 16 + (r // 32) * 4 + c.  Padding
    rows and columns hold `pad`."""
    rows, ks = s.shape
    rb, cb = (rows + 127) // 128, (K + 127) // 128
    full = torch.full((rb * 128, cb * 4), pad, dtype=torch.uint8)
    full[:rows, :ks] = s
    # (rb, r1, r0, cb, c) with row = rb*128 + r1*32 + r0, col = cb*4 + c
    t = full.view(rb, 4, 32, cb, 4).permute(0, 3, 2, 1, 4).contiguous()
    return t.view(-1)


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH[name]
