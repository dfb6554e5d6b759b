"""The C-ABI library loads without a GPU, exports every symbol include/gemm.h
declares, and rejects bad arguments before it touches a device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from dense_gemm_blackwell_sm_gb300 import build as pkg_build
from dense_gemm_blackwell_sm_gb300 import gemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


@pytest.fixture(scope="module")
def lib():
    pkg_build.build()
    return gemm.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GEMM_API\s+[\w\s\*]+?\b(gemm_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ("gemm_plan", "gemm_plan_run", "gemm_run", "gemm_run_host", "gemm_check",
                     "gemm_plan_destroy", "gemm_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(10):
        s = gemm.status_string(code)
        assert s and s != "unknown status"
    assert gemm.status_string(99) == "unknown status"
    assert "sm_103a" in gemm.version()


def _plan_status(lib, M, N, K, dtype, opts=None):
    h = ctypes.c_void_p()
    st = lib.gemm_plan(M, N, K, dtype, ctypes.byref(opts) if opts is not None else None, ctypes.byref(h))
    if h.value:
        lib.gemm_plan_destroy(h)
    return st


def test_plan_rejects_bad_sizes_without_a_device(lib):
    assert _plan_status(lib, 0, 16, 16, 0) == gemm.ERR_INVALID_ARG
    assert _plan_status(lib, 16, -1, 16, 0) == gemm.ERR_INVALID_ARG
    assert _plan_status(lib, 16, 16, 0, 0) == gemm.ERR_INVALID_ARG
    assert _plan_status(lib, 1 << 31, 16, 16, 0) == gemm.ERR_INVALID_ARG
    assert _plan_status(lib, 16, 16, 12, 0) == gemm.ERR_UNSUPPORTED_SHAPE   # K % 8 != 0
    assert _plan_status(lib, 16, 16, 16, 12) == gemm.ERR_UNSUPPORTED_DTYPE
    assert _plan_status(lib, 16, 16, 16, -1) == gemm.ERR_UNSUPPORTED_DTYPE


def test_fp8_row_pitch_rule(lib):
    # 8-bit inputs: a row of A / B is K bytes, so K must be a multiple of 16 (not 8)
    for dt in (gemm.E4M3_F32, gemm.E4M3_BF16, gemm.E5M2_F32, gemm.E5M2_BF16):
        assert _plan_status(lib, 64, 64, 24, dt) == gemm.ERR_UNSUPPORTED_SHAPE
        assert _plan_status(lib, 64, 64, 8, dt) == gemm.ERR_UNSUPPORTED_SHAPE
    assert _plan_status(lib, 64, 64, 24, gemm.BF16_BF16) != gemm.ERR_UNSUPPORTED_SHAPE
    # 8-bit inputs run on variants 7-9 only, K-major only
    assert _plan_status(lib, 64, 64, 64, gemm.E4M3_F32, gemm.make_opts(variant=gemm.S3)) == \
        gemm.ERR_UNSUPPORTED_SHAPE
    assert _plan_status(lib, 64, 64, 64, gemm.E4M3_F32, gemm.make_opts(variant=gemm.GEMV)) == \
        gemm.ERR_UNSUPPORTED_SHAPE
    assert _plan_status(lib, 64, 64, 64, gemm.E5M2_BF16,
                        gemm.make_opts(variant=gemm.S8, layout=gemm.LAYOUT_A_MN)) == gemm.ERR_UNSUPPORTED_SHAPE
    assert gemm.dtype_code("e4m3", "f32") == gemm.E4M3_F32
    assert gemm.dtype_code(torch.float8_e5m2, torch.bfloat16) == gemm.E5M2_BF16


def test_mx_rules(lib):
    for dt in (gemm.MXE4M3_F32, gemm.MXE4M3_BF16, gemm.MXE5M2_F32, gemm.MXE5M2_BF16):
        assert _plan_status(lib, 64, 64, 24, dt) == gemm.ERR_UNSUPPORTED_SHAPE
        # block-scaled inputs run on variants 7 and 8, and on 9 with bf16 C and the
        # static schedule (two consumers, 512 x 224 tiles), K-major only
        for v in (gemm.S3, gemm.S6, gemm.GEMV):
            assert _plan_status(lib, 256, 256, 256, dt, gemm.make_opts(variant=v)) == gemm.ERR_UNSUPPORTED_SHAPE
        s9 = _plan_status(lib, 256, 256, 256, dt, gemm.make_opts(variant=gemm.S9))
        if dt in (gemm.MXE4M3_F32, gemm.MXE5M2_F32):
            assert s9 == gemm.ERR_UNSUPPORTED_SHAPE
        else:
            assert s9 != gemm.ERR_UNSUPPORTED_SHAPE
            assert _plan_status(lib, 256, 256, 256, dt, gemm.make_opts(variant=gemm.S9, sched=gemm.SCHED_ATOMIC)) == \
                gemm.ERR_UNSUPPORTED_SHAPE
        assert _plan_status(lib, 256, 256, 256, dt, gemm.make_opts(variant=gemm.S7, layout=gemm.LAYOUT_A_MN)) == \
            gemm.ERR_UNSUPPORTED_SHAPE
        # the one-shot entry points have no scale arguments
        assert lib.gemm_run(64, 64, 64, 0x1000, 0x2000, 0x3000, dt, None) == gemm.ERR_INVALID_ARG
    assert lib.gemm_plan_run_mx(None, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, None, None) == gemm.ERR_INVALID_ARG
    assert gemm.dtype_code("mxe5m2", "bf16") == gemm.MXE5M2_BF16
    assert gemm.mx_scale_bytes(1, 1) == 512
    assert gemm.mx_scale_bytes(128, 128) == 512
    assert gemm.mx_scale_bytes(129, 129) == 4 * 512
    assert gemm.mx_scale_bytes(8192, 8192) == 64 * 64 * 512
    assert gemm.mx_scale_bytes(0, 128) == -1


def test_epilogue_struct_layout_matches_the_header():
    import ctypes as ct
    assert ct.sizeof(gemm.Epilogue) == 48
    assert gemm.Epilogue.scale_a.offset == 32 and gemm.Epilogue.scale_b.offset == 40


def test_plan_rejects_bad_options(lib):
    assert _plan_status(lib, 64, 64, 64, 0, gemm.make_opts(variant=12)) == gemm.ERR_INVALID_ARG
    assert _plan_status(lib, 64, 64, 64, 0, gemm.make_opts(sched=9)) == gemm.ERR_INVALID_ARG
    assert _plan_status(lib, 64, 64, 64, 0, gemm.make_opts(stages=13)) == gemm.ERR_INVALID_ARG
    # step 1 is one 128x128x64 tile; step 2 one 128x128 tile
    assert _plan_status(lib, 129, 64, 64, 0, gemm.make_opts(variant=gemm.S1)) == gemm.ERR_UNSUPPORTED_SHAPE
    assert _plan_status(lib, 64, 64, 72, 0, gemm.make_opts(variant=gemm.S1)) == gemm.ERR_UNSUPPORTED_SHAPE
    assert _plan_status(lib, 64, 200, 64, 0, gemm.make_opts(variant=gemm.S2)) == gemm.ERR_UNSUPPORTED_SHAPE
    # TMA-store writeback needs 16-byte aligned rows of C
    assert _plan_status(lib, 64, 100, 64, 3, gemm.make_opts(variant=gemm.S8)) == gemm.ERR_UNSUPPORTED_SHAPE
    assert _plan_status(lib, 17, 64, 64, 3, gemm.make_opts(variant=gemm.GEMV)) == gemm.ERR_UNSUPPORTED_SHAPE


def test_valid_plan_needs_the_device(lib):
    st = _plan_status(lib, 256, 256, 256, 3)
    if torch.cuda.is_available():
        assert st in (gemm.OK, gemm.ERR_ARCH)
    else:
        assert st == gemm.ERR_NO_DEVICE


def test_run_validates_pointers_first(lib):
    assert lib.gemm_run(64, 64, 64, None, 16, 16, 3, None) == gemm.ERR_INVALID_ARG
    assert lib.gemm_run(64, 64, 64, 0x1008, 0x2000, 0x3000, 3, None) == gemm.ERR_MISALIGNED
    assert lib.gemm_run(64, 64, 60, 0x1000, 0x2000, 0x3000, 3, None) == gemm.ERR_UNSUPPORTED_SHAPE
    assert lib.gemm_plan_run(None, 0x1000, 0x2000, 0x3000, None) == gemm.ERR_INVALID_ARG
    assert lib.gemm_plan_info(None, None) == gemm.ERR_INVALID_ARG
    lib.gemm_plan_destroy(None)   # ignored


def test_matmul_refuses_cpu_tensors(lib):
    a = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gemm.matmul(a, a)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gemm, "_lib", None)
    monkeypatch.setattr(gemm, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        gemm.load()


# The automatic plan's kernel choice, computed without a device, for a 152-SM GB300.
AUTO_CASES = [
    ((1, 4096, 4096, gemm.BF16_BF16), gemm.GEMV),       # decode GEMV, CUDA-core FMAs
    ((8, 14336, 4096, gemm.BF16_BF16), gemm.GEMV),      # decode GEMV, warp-level MMAs
    ((12, 4096, 4096, gemm.BF16_BF16), gemm.GEMV_TC),   # tcgen05 GEMV
    ((200, 100, 64, gemm.F16_BF16), gemm.S6),           # C rows of 200 B: no TMA stores
    ((8192, 8192, 8192, gemm.BF16_BF16), gemm.S9),      # 512 tiles of 512 x 256: 96 % of 7 waves
    ((8192, 14336, 4096, gemm.BF16_BF16), gemm.S9),
    ((4096, 4096, 4096, gemm.F16_F32), gemm.S9),        # (512 x 224 tiles chosen by the plan)
    ((2048, 4096, 4096, gemm.BF16_BF16), gemm.S9),      # one wave of 76 (or 64) pair tiles
    ((1024, 1024, 4096, gemm.BF16_BF16), gemm.S7),      # 32 tiles: K split 4 ways (16 pairs split 3 ways: fewer SMs)
    ((512, 4096, 4096, gemm.BF16_BF16), gemm.S8),       # 32 pair tiles: K split 2 ways
    ((1024, 1024, 1024, gemm.BF16_BF16), gemm.S7),      # too few K blocks to split; short K favours step 7
    ((256, 14336, 4096, gemm.BF16_BF16), gemm.S8),      # 56 pair tiles beat 112 single tiles
    ((1024, 4096, 4096, gemm.BF16_BF16), gemm.S8),
    ((8, 4096, 4096, gemm.E4M3_BF16), gemm.S7),         # 8-bit inputs have no GEMV (32 K blocks)
    ((8192, 8192, 8192, gemm.MXE4M3_BF16), gemm.S8),    # block-scaled, bf16 C: step 8 (step 9 on request)
    ((8192, 8192, 8192, gemm.MXE4M3_F32), gemm.S8),     # block-scaled, fp32 C: step 7 or 8
    ((128, 25600, 4096, gemm.MXE4M3_BF16), gemm.S7),    # 100 tiles: one wave of 152 CTAs, two of 76 pairs
    ((2048, 2048, 2048, gemm.BF16_BF16), gemm.S7),      # 32 K blocks: the pair's fixed cost per tile shows
    ((2048, 2048, 8192, gemm.BF16_BF16), gemm.S8),      # 128 K blocks: the pair's rate wins
    ((1024, 8192, 8192, gemm.BF16_BF16), gemm.S9),
    # short K (fewer than 32 K blocks): launch ramp and per-wave costs decide
    ((4096, 4096, 512, gemm.BF16_BF16), gemm.S7),       # 4 waves of 128 x 256 beat 2 of 512 x 224
    ((2048, 4096, 512, gemm.BF16_BF16), gemm.S7),
    ((4096, 2560, 1024, gemm.BF16_BF16), gemm.S7),      # whole tiles, no stream-K
    ((4096, 4096, 1024, gemm.BF16_BF16), gemm.S9),
    ((8192, 8192, 1024, gemm.BF16_BF16), gemm.S9),
    # few waves: stream-K on step 8's pairs beats step 9 (with or without it) from 32 K blocks
    ((4096, 2560, 2048, gemm.BF16_BF16), gemm.S8),
    ((4096, 2560, 4096, gemm.BF16_BF16), gemm.S8),
    ((2048, 5120, 2048, gemm.BF16_BF16), gemm.S8),
    ((4096, 2560, 8192, gemm.BF16_BF16), gemm.S9),      # step 9's stream-K pays from 64 K blocks
]


@pytest.mark.parametrize("args,variant", AUTO_CASES)
def test_automatic_variant_without_a_device(lib, args, variant):
    M, N, K, dt = args
    assert gemm.auto_variant(M, N, K, dt, 152) == variant


def test_automatic_variant_rejects_bad_arguments(lib):
    import ctypes
    v = ctypes.c_int32(7)
    assert lib.gemm_auto_variant(0, 16, 16, gemm.BF16_BF16, 152, ctypes.byref(v)) == gemm.ERR_INVALID_ARG
    assert v.value == 0
    assert lib.gemm_auto_variant(16, 16, 16, gemm.BF16_BF16, 1, ctypes.byref(v)) == gemm.ERR_INVALID_ARG
    assert lib.gemm_auto_variant(16, 16, 16, 99, 152, ctypes.byref(v)) == gemm.ERR_UNSUPPORTED_DTYPE
    assert lib.gemm_auto_variant(16, 16, 12, gemm.BF16_BF16, 152, ctypes.byref(v)) == gemm.ERR_UNSUPPORTED_SHAPE
    assert lib.gemm_auto_variant(16, 16, 16, gemm.BF16_BF16, 152, None) == gemm.ERR_INVALID_ARG
