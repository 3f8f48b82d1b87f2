"""ctypes declarations of the C ABI in include/moe_plan.h.

Loading fails loudly when the CUDA library has not been built: there is no
other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_GB300_LIB names another build of the same library (e.g. one compiled
# with different options); by default the in-tree build is loaded.
LIB_PATH = os.environ.get("MOE_GB300_LIB") or os.path.join(PKG, "libmoe_gb300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moe_plan.h")

MOE_OK, MOE_EINVAL, MOE_EALIGN, MOE_ECUDA = 0, 1, 2, 3
MOE_BF16, MOE_F32, MOE_FP8_E4M3 = 0, 1, 2

P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "moe_version": (I32, []),
    "moe_status_string": (ctypes.c_char_p, [I32]),
    "moe_last_cuda_error": (I32, []),
    "moe_plan_workspace_size": (SZ, [I64, I32, I32]),
    "moe_plan": (I32, [P, I64, I32, I32, P, P, P, P, P, P, SZ, P]),
    "moe_plan_static_scratch": (I32, [P, I64, I32, I32, P, P, P, P, P, P]),
    "moe_plan_capacity": (I32, [P, I64, I32, I32, I64, P, P, P, P, P, P, P, SZ, P]),
    "moe_group_plan_workspace_size": (SZ, [I64, I32, I32, I32]),
    "moe_group_plan": (I32, [P, P, I64, I32, I32, I32, P, P, P, P, P, P, SZ, P]),
    "moe_dispatch": (I32, [P, I64, I64, I32, I32, P, P, I64, P, I64, P, P]),
    "moe_dispatch_dedup": (I32, [P, I64, I64, I32, I32, I32, P, P, P, P, I64, P, P, I64, P]),
    "moe_dispatch_quant_fp8": (I32, [P, I64, I64, I32, P, I32, P, P, I64, P]),
    "moe_combine": (I32, [P, I64, I32, P, P, I64, I64, I32, P, I32, P]),
    "moe_combine_dedup": (I32, [P, I64, I32, P, P, I32, P, P, P, I64, I64, I32, I64, P, P, I32,
                                P]),
    "moe_combine_fold": (I32, [P, I64, I32, P, I32, P, I64, I64, I32, P, I32, P, P]),
    "moe_plan_dispatch_fused_max": (I64, []),
    "moe_plan_dispatch": (I32, [P, P, I64, I64, I32, I32, I32, P, I64, P, P, P, P, P, P, I64, P,
                                P, SZ, P]),
    "moe_device_errors": (I32, [P]),
    "moe_selftest_wait_timeout": (I32, [I64, P]),
    "moe_selftest_convert": (I32, [ctypes.c_uint32, I64, P, P, P]),
}

_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        msg = f"{fn}: status {status}"
        lib = _lib
        if lib is not None:
            msg += f" ({lib.moe_status_string(status).decode()})"
        if status == MOE_ECUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


def load() -> ctypes.CDLL:
    """Load libmoe_gb300.so (built by combine_moe_plan_02_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -m combine_moe_plan_02_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER):
    """Names of the functions declared in the public header."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status, _lib.moe_last_cuda_error() if _lib is not None else 0)
