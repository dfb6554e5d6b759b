"""GB300 (sm_103a) dense GEMM C = A * B^T and decode GEMV behind a C ABI.

The kernels live in libdgbgemm.so (built from csrc/ by ``build.build()``);
``gemm`` is its ctypes binding.  Importing the package does not load the
library; the first call does, and raises if it is missing.
"""
from .gemm import (GemmError, Plan, PlanInfo, Opts, load, make_opts, matmul, gemm_run, gemm_run_host,  # noqa: F401
                   gemm_check, dtype_code, status_string, version)

__all__ = ["GemmError", "Plan", "PlanInfo", "Opts", "load", "make_opts", "matmul", "gemm_run",
           "gemm_run_host", "gemm_check", "dtype_code", "status_string", "version"]
