"""ctypes binding of the C ABI in include/gemm.h (argument marshalling only).

Every computation happens inside libdgbgemm.so's CUDA kernels; this module
only converts torch tensors / integers into the pointers and sizes the C
functions take, and status codes into exceptions.  There is no fallback: if
the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdgbgemm.so")

# gemm_dtype_t
F16_F32, F16_BF16, BF16_F32, BF16_BF16 = 0, 1, 2, 3
E4M3_F32, E4M3_BF16, E5M2_F32, E5M2_BF16 = 4, 5, 6, 7
MXE4M3_F32, MXE4M3_BF16, MXE5M2_F32, MXE5M2_BF16 = 8, 9, 10, 11
DTYPES = {("f16", "f32"): F16_F32, ("f16", "bf16"): F16_BF16,
          ("bf16", "f32"): BF16_F32, ("bf16", "bf16"): BF16_BF16,
          ("e4m3", "f32"): E4M3_F32, ("e4m3", "bf16"): E4M3_BF16,
          ("e5m2", "f32"): E5M2_F32, ("e5m2", "bf16"): E5M2_BF16,
          ("mxe4m3", "f32"): MXE4M3_F32, ("mxe4m3", "bf16"): MXE4M3_BF16,
          ("mxe5m2", "f32"): MXE5M2_F32, ("mxe5m2", "bf16"): MXE5M2_BF16}

# gemm_status_t
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_UNSUPPORTED_DTYPE = 0, 1, 2, 3, 4
ERR_ARCH, ERR_CUDA, ERR_OOM, ERR_DEVICE_TIMEOUT, ERR_NO_DEVICE = 5, 6, 7, 8, 9

# gemm_variant_t
VARIANT_AUTO, S1, S2, S3, S4, S5, S6, S7, S8, S9, GEMV, GEMV_TC = range(12)
VARIANT_NAMES = {0: "auto", 1: "s1_single_tile", 2: "s2_kloop", 3: "s3_multi_cta", 4: "s4_tma",
                 5: "s5_pipeline", 6: "s6_persistent", 7: "s7_warp_specialized", 8: "s8_cta_pair",
                 9: "s9_two_consumers", 10: "gemv", 11: "gemv_tc"}

# gemm_sched_t
SCHED_AUTO, SCHED_STATIC, SCHED_ATOMIC, SCHED_CLC, SCHED_STREAM_K = 0, 1, 2, 3, 4

# gemm_activation_t
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU_TANH, ACT_GELU_ERF = 0, 1, 2, 3, 4

DEBUG_SKIP_ONE_LOAD = 1
FLAG_STATIC_B = 1
LAYOUT_A_MN, LAYOUT_B_MN = 1, 2


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class Opts(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("sched", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("raster_group", ctypes.c_int32), ("max_ctas", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("timeout_ns", ctypes.c_int64), ("debug_flags", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32 * 5)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("variant", "sched", "stages", "raster_group", "tile_m", "tile_n",
                                              "cluster", "consumers", "grid", "smem_bytes", "num_sms", "tiles",
                                              "narrow_tile_n", "wide_cols")]

    def as_dict(self) -> dict:
        d = {n: int(getattr(self, n)) for n, _ in self._fields_}
        d["variant_name"] = VARIANT_NAMES.get(d["variant"], "?")
        return d


class Epilogue(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p), ("activation", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 3), ("scale_a", ctypes.c_void_p), ("scale_b", ctypes.c_void_p)]


_lib = None


def load():
    """Load libdgbgemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdgbgemm.so is not built (%s); run __graft_entry__.build() first" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.gemm_plan.argtypes = [i64, i64, i64, i32, ctypes.POINTER(Opts), ctypes.POINTER(p)]
    lib.gemm_plan.restype = i32
    lib.gemm_plan_run.argtypes = [p, p, p, p, p]
    lib.gemm_plan_run.restype = i32
    lib.gemm_plan_run_epilogue.argtypes = [p, p, p, p, ctypes.POINTER(Epilogue), p]
    lib.gemm_plan_run_epilogue.restype = i32
    lib.gemm_plan_run_mx.argtypes = [p, p, p, p, p, p, ctypes.POINTER(Epilogue), p]
    lib.gemm_plan_run_mx.restype = i32
    lib.gemm_mx_scale_bytes.argtypes = [i64, i64]
    lib.gemm_mx_scale_bytes.restype = i64
    lib.gemm_auto_variant.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(i32)]
    lib.gemm_auto_variant.restype = i32
    lib.gemm_run.argtypes = [i64, i64, i64, p, p, p, i32, p]
    lib.gemm_run.restype = i32
    lib.gemm_run_host.argtypes = [i64, i64, i64, p, p, p, i32, p, p, p, p]
    lib.gemm_run_host.restype = i32
    lib.gemm_check.argtypes = [p, p]
    lib.gemm_check.restype = i32
    lib.gemm_plan_info.argtypes = [p, ctypes.POINTER(PlanInfo)]
    lib.gemm_plan_info.restype = i32
    lib.gemm_plan_set_visits.argtypes = [p, p]
    lib.gemm_plan_set_visits.restype = i32
    lib.gemm_plan_destroy.argtypes = [p]
    lib.gemm_plan_destroy.restype = None
    lib.gemm_clear_cache.argtypes = []
    lib.gemm_clear_cache.restype = None
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_version.argtypes = []
    lib.gemm_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise GemmError(status, where)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def make_opts(variant=0, sched=0, stages=0, raster_group=0, max_ctas=0, timeout_ns=0, debug_flags=0,
              split_k=0, flags=0, layout=0) -> Opts:
    o = Opts()
    o.flags = int(flags)
    o.layout = int(layout)
    o.split_k = int(split_k)
    o.variant, o.sched, o.stages, o.raster_group = int(variant), int(sched), int(stages), int(raster_group)
    o.max_ctas, o.timeout_ns, o.debug_flags = int(max_ctas), int(timeout_ns), int(debug_flags)
    return o


class Plan:
    """A plan for C = A * B^T of fixed sizes and dtypes (gemm_plan)."""

    def __init__(self, M: int, N: int, K: int, dtype: int, opts: Opts | None = None):
        lib = load()
        h = ctypes.c_void_p()
        st = lib.gemm_plan(int(M), int(N), int(K), int(dtype), ctypes.byref(opts) if opts is not None else None,
                           ctypes.byref(h))
        _check(st, "gemm_plan")
        self._h = h
        self.M, self.N, self.K, self.dtype = int(M), int(N), int(K), int(dtype)

    def run_ptr(self, a_ptr: int, b_ptr: int, c_ptr: int, stream_ptr: int = 0) -> int:
        return load().gemm_plan_run(self._h, a_ptr, b_ptr, c_ptr, stream_ptr)

    def run(self, a, b, c, stream=None):
        _check(self.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), _stream_ptr(stream)), "gemm_plan_run")
        return c

    def run_epilogue(self, a, b, c, bias=None, residual=None, act: int = ACT_NONE, stream=None,
                     scale_a=None, scale_b=None):
        """C = act(scale_a[:, None] * scale_b[None, :] * (a @ b.T) + bias) + residual in one
        kernel (variants 7-9).  bias, scale_b: fp32 CUDA tensors of N values; scale_a: M values;
        residual: (M, N) CUDA tensor of C's type."""
        e = Epilogue()
        e.scale_a = None if scale_a is None else scale_a.data_ptr()
        e.scale_b = None if scale_b is None else scale_b.data_ptr()
        e.bias = None if bias is None else bias.data_ptr()
        e.residual = None if residual is None else residual.data_ptr()
        e.activation = int(act)
        st = load().gemm_plan_run_epilogue(self._h, a.data_ptr(), b.data_ptr(), c.data_ptr(), ctypes.byref(e),
                                           _stream_ptr(stream))
        _check(st, "gemm_plan_run_epilogue")
        return c

    def run_mx(self, a, b, c, sf_a, sf_b, bias=None, residual=None, act=None, stream=None,
               scale_a=None, scale_b=None):
        """Block-scaled C = (X_A . a) @ (X_B . b).T for a plan of an MX dtype: sf_a / sf_b
        are uint8 CUDA tensors of UE8M0 scales in the tiled layout (mx_scale_bytes(rows, K)
        bytes each).  With any of bias / residual / act / scale_a / scale_b the fused
        epilogue runs as in run_epilogue."""
        e = None
        if bias is not None or residual is not None or act is not None or scale_a is not None or \
                scale_b is not None:
            e = Epilogue()
            e.bias = None if bias is None else bias.data_ptr()
            e.residual = None if residual is None else residual.data_ptr()
            e.activation = int(act or ACT_NONE)
            e.scale_a = None if scale_a is None else scale_a.data_ptr()
            e.scale_b = None if scale_b is None else scale_b.data_ptr()
        st = load().gemm_plan_run_mx(self._h, a.data_ptr(), b.data_ptr(), c.data_ptr(), sf_a.data_ptr(),
                                     sf_b.data_ptr(), None if e is None else ctypes.byref(e), _stream_ptr(stream))
        _check(st, "gemm_plan_run_mx")
        return c

    def check(self, stream=None) -> int:
        return load().gemm_check(self._h, _stream_ptr(stream))

    def info(self) -> dict:
        inf = PlanInfo()
        _check(load().gemm_plan_info(self._h, ctypes.byref(inf)), "gemm_plan_info")
        return inf.as_dict()

    def set_visits(self, visits) -> None:
        _check(load().gemm_plan_set_visits(self._h, None if visits is None else visits.data_ptr()),
               "gemm_plan_set_visits")

    def destroy(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            load().gemm_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def dtype_code(in_dtype, out_dtype) -> int:
    import torch
    names = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32",
             torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}
    i = names.get(in_dtype, in_dtype)
    o = names.get(out_dtype, out_dtype)
    if (i, o) not in DTYPES:
        raise ValueError("unsupported dtype pair %r -> %r" % (i, o))
    return DTYPES[(i, o)]


def auto_variant(M: int, N: int, K: int, dtype: int, num_sms: int) -> int:
    """The variant the automatic plan takes on a GPU with num_sms SMs (gemm_auto_variant);
    needs no device.  Raises GemmError for invalid arguments."""
    v = ctypes.c_int32(0)
    _check(load().gemm_auto_variant(int(M), int(N), int(K), int(dtype), int(num_sms), ctypes.byref(v)),
           "gemm_auto_variant")
    return int(v.value)


def mx_scale_bytes(rows: int, K: int) -> int:
    """Bytes of one tiled MX scale array (gemm_mx_scale_bytes)."""
    return int(load().gemm_mx_scale_bytes(int(rows), int(K)))


def gemm_run(M, N, K, a_ptr, b_ptr, c_ptr, dtype, stream_ptr=0) -> int:
    return load().gemm_run(int(M), int(N), int(K), a_ptr, b_ptr, c_ptr, int(dtype), stream_ptr)


def gemm_run_host(M, N, K, a_host_ptr, b_host_ptr, c_host_ptr, dtype, da, db, dc, stream_ptr=0) -> int:
    return load().gemm_run_host(int(M), int(N), int(K), a_host_ptr, b_host_ptr, c_host_ptr, int(dtype),
                                da, db, dc, stream_ptr)


def gemm_check(stream=None) -> int:
    return load().gemm_check(None, _stream_ptr(stream))


_layout_plans: dict = {}


def _stored(x):
    """(tensor as stored, is_mn_major) for a logical (rows x K) operand: a
    contiguous tensor is K-major; a transposed view of a contiguous K x rows
    tensor is passed as stored, MN-major, without a copy."""
    if x.is_contiguous():
        return x, False
    if x.t().is_contiguous():
        return x.t(), True
    return x.contiguous(), False


def matmul(a, b, out_dtype=None, out=None, stream=None):
    """C = a @ b.T for CUDA tensors a (M x K) and b (N x K), fp16, bf16,
    float8_e4m3fn or float8_e5m2.

    ``out_dtype`` is torch.float32 (default) or torch.bfloat16.  A 16-bit operand
    that is the transpose of a contiguous tensor (``x.t()``) is read in place as
    an MN-major operand by the warp-specialised kernels; 8-bit operands are
    K-major only and are made contiguous first.
    """
    import torch
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("matmul takes CUDA tensors")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("shapes must be (M, K) and (N, K)")
    if a.dtype != b.dtype:
        raise ValueError("a and b must share a dtype")
    out_dtype = out_dtype or (out.dtype if out is not None else torch.float32)
    code = dtype_code(a.dtype, out_dtype)
    M, K = a.shape
    N = b.shape[0]
    a_s, a_mn = _stored(a)
    b_s, b_mn = _stored(b)
    if out is None:
        out = torch.empty((M, N), device=a.device, dtype=out_dtype)
    elif out.shape != (M, N) or not out.is_contiguous() or out.dtype != out_dtype:
        raise ValueError("out must be a contiguous (M, N) tensor of out_dtype")
    layout = (LAYOUT_A_MN if a_mn else 0) | (LAYOUT_B_MN if b_mn else 0)
    if layout and ((a_mn and M % 8) or (b_mn and N % 8) or a.element_size() == 1):
        a_s, b_s, layout = a.contiguous(), b.contiguous(), 0
    if layout == 0:
        _check(gemm_run(M, N, K, a_s.data_ptr(), b_s.data_ptr(), out.data_ptr(), code, _stream_ptr(stream)),
               "gemm_run")
        return out
    key = (M, N, K, code, layout, a.device.index)
    plan = _layout_plans.get(key)
    if plan is None:
        plan = _layout_plans[key] = Plan(M, N, K, code, make_opts(layout=layout))
    _check(plan.run_ptr(a_s.data_ptr(), b_s.data_ptr(), out.data_ptr(), _stream_ptr(stream)), "gemm_plan_run")
    return out


def version() -> str:
    return load().gemm_version().decode()
