"""gemm_run_noalloc, the entry point for callers that must not allocate memory
(allocator hooks, out-of-memory handlers, locked memory pools, embedders with
pre-assigned memory), called through the C ABI.

Its results must agree with gemm_run's -- within the per-element tolerance of
the parity tests, S = sum_k |a_ik b_jk| coming from the CPU oracle -- on calls
made one right after the other, which share the library's fixed scratch array
(so each call must clear what the previous one left there).  The shapes take
the 128x256, 256x256 and 512x256 tile paths.  The first test makes the entry
point's first call on the device before any gemm_run, and checks that a later
call changes neither torch's allocated bytes nor the device's free memory.
This file is collected last, and passes both alone in a fresh process and
after the other tests.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (M, N, K, in, out, seed): 128x256 tiles, 256x256 CTA-pair tiles, 512x256 two-consumer tiles
CALLS = [(600, 776, 264, "bf16", "bf16", 1), (2048, 2560, 128, "bf16", "bf16", 2),
         (4096, 4096, 128, "f16", "f32", 3)]


@pytest.fixture(scope="module")
def noalloc():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    lib = gemm.load()
    f = lib.gemm_run_noalloc
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def test_first_call_sets_up_and_later_calls_allocate_nothing(noalloc):
    """The first call on a device resolves the scratch array and loads every
    kernel the entry point can launch (it may let the driver reserve memory for
    code); every later call -- including the first with another output type and
    tile -- must leave device memory exactly as it was."""
    stream = torch.cuda.current_stream().cuda_stream
    M, N, K = 700, 1288, 264
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("normal", 1.0), seed=7)
    da, db = a.to(DEV), b.to(DEV)
    c16 = torch.full((M, N), float("nan"), device=DEV, dtype=torch.bfloat16)
    c32 = torch.full((M, N), float("nan"), device=DEV, dtype=torch.float32)
    # a shape for the 512 x 256 tile: outputs allocated before anything is measured
    M2, N2, K2 = 4096, 4096, 128
    a2, b2 = inputs.make_operands(M2, N2, K2, "bf16", ("uniform",), ("normal", 1.0), seed=8)
    da2, db2 = a2.to(DEV), b2.to(DEV)
    c2 = torch.full((M2, N2), float("nan"), device=DEV, dtype=torch.float32)
    assert noalloc(M, N, K, da.data_ptr(), db.data_ptr(), c16.data_ptr(), gemm.BF16_BF16, stream) == gemm.OK
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    assert noalloc(M, N, K, da.data_ptr(), db.data_ptr(), c32.data_ptr(), gemm.BF16_F32, stream) == gemm.OK
    assert noalloc(M2, N2, K2, da2.data_ptr(), db2.data_ptr(), c2.data_ptr(), gemm.BF16_F32, stream) == gemm.OK
    assert noalloc(M, N, K, da.data_ptr(), db.data_ptr(), c16.data_ptr(), gemm.BF16_BF16, stream) == gemm.OK
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    assert after == before
    ref, S = oracle.gemm(a, b)
    assert parity.check(c16.double().cpu().numpy(), ref, S, "bf16")["ok"]
    assert parity.check(c32.double().cpu().numpy(), ref, S, "f32")["ok"]
    ref2, S2 = oracle.gemm(a2, b2)
    assert parity.check(c2.double().cpu().numpy(), ref2, S2, "f32")["ok"]


def test_noalloc_agrees_with_gemm_run_on_consecutive_calls(noalloc):
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K, ti, to, seed in CALLS:
        a, b = inputs.make_operands(M, N, K, ti, ("uniform",), ("normal", 1.0), seed=seed)
        da, db = a.to(DEV), b.to(DEV)
        code = gemm.dtype_code(ti, to)
        out_t = inputs.torch_dtype(to)
        c_run = torch.empty((M, N), device=DEV, dtype=out_t)
        assert gemm.gemm_run(M, N, K, da.data_ptr(), db.data_ptr(), c_run.data_ptr(), code, stream) == gemm.OK
        c_na = torch.full((M, N), float("nan"), device=DEV, dtype=out_t)
        assert noalloc(M, N, K, da.data_ptr(), db.data_ptr(), c_na.data_ptr(), code, stream) == gemm.OK
        torch.cuda.synchronize()
        assert gemm.gemm_check() == gemm.OK
        ref, S = oracle.gemm(a, b)
        x = c_na.double().cpu().numpy()
        y = c_run.double().cpu().numpy()
        assert np.isfinite(x).all()
        tol = parity.bound(y, S, to)
        bad = np.argwhere(np.abs(x - y) > tol)
        assert bad.size == 0, ((M, N, K), bad[:3])
        assert parity.check(x, ref, S, to)["ok"]


def test_noalloc_rejects_bad_arguments(noalloc):
    stream = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    assert noalloc(64, 64, 60, a.data_ptr(), a.data_ptr(), a.data_ptr(), gemm.BF16_BF16, stream) == \
        gemm.ERR_UNSUPPORTED_SHAPE
    assert noalloc(64, 100, 64, a.data_ptr(), a.data_ptr(), a.data_ptr(), gemm.BF16_BF16, stream) == \
        gemm.ERR_UNSUPPORTED_SHAPE
    assert noalloc(64, 64, 64, None, a.data_ptr(), a.data_ptr(), gemm.BF16_BF16, stream) == gemm.ERR_INVALID_ARG
    assert noalloc(64, 64, 64, a.data_ptr() + 2, a.data_ptr(), a.data_ptr(), gemm.BF16_BF16, stream) == \
        gemm.ERR_MISALIGNED
    assert noalloc(64, 64, 64, a.data_ptr(), a.data_ptr(), a.data_ptr(), 9, stream) == gemm.ERR_UNSUPPORTED_DTYPE
