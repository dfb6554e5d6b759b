"""CPU oracle for C = A * B^T -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import this package.  The product (``dense_gemm_blackwell_sm_gb300``)
never imports it, and the two share no code: the arithmetic lives in
``gemm_oracle.c`` (plain fp64 triple loop, OpenMP over rows), built into
``liboracle.so`` next to it by :func:`build`.

Every function here is the plain definition
``C[i,j] = sum_k a[i,k] * b[j,k]`` (with ``S[i,j] = sum_k |a[i,k] * b[j,k]|``)
of the dense GEMM that "Modern GPU Programming for MLSys" (reading notes,
section "9 步优化", steps 1-3) computes tile by tile; see the C file's header.

Pins (tests/test_oracle_pins.py): exact-rational brute force on tiny shapes,
identity / permutation operands, the rank-1 closed form, transpose symmetry,
additivity, thread-count invariance and an exhaustive check of both 16-bit
decoders against numpy's IEEE binary16 / binary32 conversions.  The fused
epilogue (``epilogue``: bias, activation, residual) is pinned in
tests/test_oracle_epilogue_pins.py; the 8-bit float inputs (E4M3 / E5M2), the
dequantisation scales and the MX block-scaled product (``gemm_mx``) in
tests/test_oracle_fp8_pins.py and tests/test_oracle_mx_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

IN_F16 = 0
IN_BF16 = 1
IN_E4M3 = 2
IN_E5M2 = 3

_lib = None


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm_rows_f64.argtypes = [i64, i64, i64, p, p, ctypes.c_int,
                                             p, i64, p, p, ctypes.c_int]
        lib.oracle_gemm_rows_f64.restype = ctypes.c_int
        lib.oracle_gemm_f64.argtypes = [i64, i64, i64, p, p, ctypes.c_int, p, p, ctypes.c_int]
        lib.oracle_gemm_f64.restype = ctypes.c_int
        lib.oracle_widen.argtypes = [ctypes.c_uint16, ctypes.c_int]
        lib.oracle_widen.restype = ctypes.c_double
        lib.oracle_gemm8_rows_f64.argtypes = [i64, i64, i64, p, p, ctypes.c_int, p, i64, p, p, ctypes.c_int]
        lib.oracle_gemm8_rows_f64.restype = ctypes.c_int
        lib.oracle_widen8.argtypes = [ctypes.c_uint8, ctypes.c_int]
        lib.oracle_widen8.restype = ctypes.c_double
        lib.oracle_gemm_mx_rows_f64.argtypes = [i64, i64, i64, p, p, ctypes.c_int, p, p, p, i64, p, p,
                                                 ctypes.c_int]
        lib.oracle_gemm_mx_rows_f64.restype = ctypes.c_int
        lib.oracle_ue8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_ue8m0.restype = ctypes.c_double
        lib.oracle_scale_f64.argtypes = [i64, i64, p, p, p]
        lib.oracle_scale_f64.restype = ctypes.c_int
        lib.oracle_epilogue_f64.argtypes = [i64, i64, p, p, p, ctypes.c_int, ctypes.c_int]
        lib.oracle_epilogue_f64.restype = ctypes.c_int
        lib.oracle_activation.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.oracle_activation.restype = ctypes.c_double
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """Raw 16-bit patterns of a 2-D fp16/bf16 array (torch tensor or uint16 ndarray)."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.float16:
            x = x.view(np.uint16)
        if x.dtype != np.uint16:
            raise TypeError("oracle operands must be 16-bit patterns")
        return np.ascontiguousarray(x)
    import torch  # only for tensor inputs
    if x.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("oracle operands must be fp16 or bf16")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def kind_of(x) -> int:
    """IN_F16, IN_BF16, IN_E4M3 or IN_E5M2 for a torch tensor / numpy array."""
    if isinstance(x, np.ndarray):
        return IN_F16
    import torch
    if x.dtype == torch.float8_e4m3fn:
        return IN_E4M3
    if x.dtype == torch.float8_e5m2:
        return IN_E5M2
    return IN_BF16 if x.dtype == torch.bfloat16 else IN_F16


def _bytes8(x) -> np.ndarray:
    """Raw 8-bit patterns of a 2-D fp8 array (torch tensor or uint8 ndarray)."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint8:
            raise TypeError("8-bit operands must be uint8 patterns")
        return np.ascontiguousarray(x)
    import torch
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.uint8).numpy())


def widen8(bits: int, kind: int) -> float:
    """Exact value of one 8-bit pattern (kind IN_E4M3 or IN_E5M2)."""
    return float(_load().oracle_widen8(int(bits) & 0xFF, int(kind)))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def widen(bits: int, kind: int) -> float:
    """Exact value of one 16-bit pattern (kind IN_F16 or IN_BF16)."""
    return float(_load().oracle_widen(int(bits) & 0xFFFF, int(kind)))


def _gemm8(a, b, kind, rows, nthreads):
    A, B = _bytes8(a), _bytes8(b)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = M if r is None else len(r)
    C = np.empty((n, N), dtype=np.float64)
    S = np.empty((n, N), dtype=np.float64)
    rc = _load().oracle_gemm8_rows_f64(M, N, K, A.ctypes.data, B.ctypes.data, kind,
                                       None if r is None else r.ctypes.data, n, C.ctypes.data,
                                       S.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm8_rows_f64 rejected its arguments")
    return C, S


def _u8(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x.astype(np.uint8, copy=False))
    import torch
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.uint8).numpy())


def ue8m0(e: int) -> float:
    """Value of one UE8M0 scale byte: 2^(e - 127), NaN for 255."""
    return float(_load().oracle_ue8m0(int(e) & 0xFF))


def gemm_mx(a, b, scale_a, scale_b, rows=None, kind: int | None = None, nthreads: int = 0):
    """MX block-scaled product of 8-bit operands, in fp64:
    C[i,j] = sum_k (X_A[i,k//32] a[i,k]) (X_B[j,k//32] b[j,k]), with S the sum of
    the terms' magnitudes.  scale_a (M x ceil(K/32)) and scale_b (N x ceil(K/32))
    hold UE8M0 bytes, row-major.  ``rows`` restricts C and S to those rows of A."""
    kind = kind_of(a) if kind is None else kind
    if kind not in (IN_E4M3, IN_E5M2):
        raise ValueError("MX block scaling takes 8-bit float operands")
    A, B = _bytes8(a), _bytes8(b)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    SA, SB = _u8(scale_a), _u8(scale_b)
    ks = (K + 31) // 32
    if SA.shape != (M, ks) or SB.shape != (N, ks):
        raise ValueError("scales must be M x ceil(K/32) and N x ceil(K/32)")
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = M if r is None else len(r)
    C = np.empty((n, N), dtype=np.float64)
    S = np.empty((n, N), dtype=np.float64)
    rc = _load().oracle_gemm_mx_rows_f64(M, N, K, A.ctypes.data, B.ctypes.data, kind, SA.ctypes.data,
                                         SB.ctypes.data, None if r is None else r.ctypes.data, n,
                                         C.ctypes.data, S.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_mx_rows_f64 rejected its arguments")
    return C, S


def gemm(a, b, kind: int | None = None, nthreads: int = 0):
    """Full fp64 C = A * B^T and S = sum_k |a_ik b_jk|; returns (C, S) as float64 arrays."""
    kind = kind_of(a) if kind is None else kind
    if kind in (IN_E4M3, IN_E5M2):
        return _gemm8(a, b, kind, None, nthreads)
    A, B = _bits(a), _bits(b)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_f64(M, N, K, A.ctypes.data, B.ctypes.data, kind,
                                 C.ctypes.data, S.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_f64 rejected its arguments")
    return C, S


def gemm_rows(a, b, rows, kind: int | None = None, nthreads: int = 0):
    """Rows ``rows`` of C and S only (len(rows) x N each)."""
    kind = kind_of(a) if kind is None else kind
    if kind in (IN_E4M3, IN_E5M2):
        return _gemm8(a, b, kind, rows, nthreads)
    A, B = _bits(a), _bits(b)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    C = np.empty((len(r), N), dtype=np.float64)
    S = np.empty((len(r), N), dtype=np.float64)
    rc = _load().oracle_gemm_rows_f64(M, N, K, A.ctypes.data, B.ctypes.data, kind,
                                      r.ctypes.data, len(r), C.ctypes.data, S.ctypes.data,
                                      int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_rows_f64 rejected its arguments")
    return C, S


ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU_TANH, ACT_GELU_ERF = 0, 1, 2, 3, 4


def activation(x: float, act: int) -> float:
    """The oracle's activation of one value (fp64)."""
    return float(_load().oracle_activation(float(x), int(act)))


def _f32_vector(v, n: int, what: str):
    if v is None:
        return None
    if hasattr(v, "detach"):
        v = v.detach().cpu().numpy()
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    if a.shape != (n,):
        raise ValueError("%s must hold %d values" % (what, n))
    return a


def scale(C, scale_a=None, scale_b=None):
    """C[i][j] * scale_a[i] * scale_b[j] in fp64, on a copy of C (M x N); the
    scales are fp32 vectors (array or tensor) of M and N values, or None."""
    out = np.ascontiguousarray(np.array(C, dtype=np.float64))
    M, N = out.shape
    sa = _f32_vector(scale_a, M, "scale_a")
    sb = _f32_vector(scale_b, N, "scale_b")
    rc = _load().oracle_scale_f64(M, N, out.ctypes.data, None if sa is None else sa.ctypes.data,
                                  None if sb is None else sb.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_scale_f64 rejected its arguments")
    return out


def epilogue(C, bias=None, residual=None, act: int = ACT_NONE, scale_a=None, scale_b=None):
    """act(scale_a[row] * scale_b[col] * C + bias[col]) + residual, in fp64, on a
    copy of C (M x N).

    bias, scale_b: N fp32 values (array or tensor) or None; scale_a: M fp32
    values or None; residual: M x N fp32 / bf16 / fp16 (numpy float32 array, or
    torch tensor) or None."""
    out = np.ascontiguousarray(np.array(C, dtype=np.float64))
    if scale_a is not None or scale_b is not None:
        out = scale(out, scale_a, scale_b)
    M, N = out.shape
    b = None
    if bias is not None:
        if hasattr(bias, "detach"):
            bias = bias.detach().cpu().numpy()
        b = np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
        if b.shape != (N,):
            raise ValueError("bias must hold N values")
    r, kind = None, 0
    if residual is not None:
        if hasattr(residual, "detach"):
            import torch
            t = residual.detach().cpu().contiguous()
            if t.dtype == torch.float32:
                r, kind = t.numpy(), 1
            else:
                r, kind = _bits(t), (2 if t.dtype == torch.bfloat16 else 3)
        else:
            r, kind = np.ascontiguousarray(np.asarray(residual, dtype=np.float32)), 1
        if r.shape != (M, N):
            raise ValueError("residual must be M x N")
    rc = _load().oracle_epilogue_f64(M, N, out.ctypes.data, None if b is None else b.ctypes.data,
                                     None if r is None else r.ctypes.data, kind, int(act))
    if rc != 0:
        raise ValueError("oracle_epilogue_f64 rejected its arguments")
    return out
