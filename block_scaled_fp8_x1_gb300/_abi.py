"""ctypes declarations of libfp8rl's C ABI (``include/fp8rl.h``).

Loading fails loudly when the shared library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8rl.so")

STATUS_NAMES = {
    0: "FP8RL_OK",
    1: "FP8RL_ERR_INVALID_ARG",
    2: "FP8RL_ERR_SHAPE",
    3: "FP8RL_ERR_ALIGN",
    4: "FP8RL_ERR_UNSUPPORTED_DEVICE",
    5: "FP8RL_ERR_WORKSPACE",
    6: "FP8RL_ERR_CUDA",
    7: "FP8RL_ERR_DEVICE_TIMEOUT",
    8: "FP8RL_ERR_DEVICE_BOUNDS",
}
FP8RL_OK = 0
FP8RL_ERR_INVALID_ARG = 1
FP8RL_ERR_SHAPE = 2
FP8RL_ERR_ALIGN = 3
FP8RL_ERR_UNSUPPORTED_DEVICE = 4
FP8RL_ERR_WORKSPACE = 5
FP8RL_ERR_CUDA = 6
FP8RL_ERR_DEVICE_TIMEOUT = 7
FP8RL_ERR_DEVICE_BOUNDS = 8

FP8RL_OP_FWD, FP8RL_OP_DGRAD, FP8RL_OP_WGRAD = 0, 1, 2
FP8RL_VARIANT_AUTO, FP8RL_VARIANT_TILED, FP8RL_VARIANT_SPLITK, FP8RL_VARIANT_PAIR = 0, 1, 2, 3
FP8RL_VARIANT_DECODE = 4
FP8RL_VARIANT_MULTICAST = 5


class Fp8rlError(RuntimeError):
    """A libfp8rl entry point returned a status other than FP8RL_OK."""

    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


class GemmOpts(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("splits", ctypes.c_int), ("grid", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("epi_warps", ctypes.c_int)]


P = ctypes.c_void_p
I64 = ctypes.c_int64
ST = ctypes.c_int
STREAM = ctypes.c_void_p

# name -> (restype, argtypes); the order follows include/fp8rl.h
SIGNATURES = {
    "fp8rl_version": (ctypes.c_int, []),
    "fp8rl_status_string": (ctypes.c_char_p, [ST]),
    "fp8rl_init": (ST, [ctypes.c_int]),
    "fp8rl_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "fp8rl_check_status": (ST, [STREAM]),
    "fp8rl_quantize_1x128": (ST, [P, I64, I64, I64, P, P, P, P, STREAM]),
    "fp8rl_quantize_128x1": (ST, [P, I64, I64, I64, P, P, STREAM]),
    "fp8rl_requantize_128x1": (ST, [P, P, I64, I64, P, P, STREAM]),
    "fp8rl_quantize_128x128": (ST, [P, I64, I64, I64, P, P, P, STREAM]),
    "fp8rl_rmsnorm_quant": (ST, [P, P, ctypes.c_float, I64, I64, P, P, P, P, P, STREAM]),
    "fp8rl_silu_mul_quant": (ST, [P, I64, I64, P, P, P, P, STREAM]),
    "fp8rl_silu_mul_bwd_quant": (ST, [P, P, I64, I64, P, P, P, P, STREAM]),
    "fp8rl_rmsnorm_bwd": (ST, [P, P, P, P, I64, I64, P, P, P, ctypes.c_size_t, STREAM]),
    "fp8rl_rmsnorm_bwd_workspace_bytes": (ctypes.c_size_t, [I64, I64]),
    "fp8rl_gemm_fwd": (ST, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t, STREAM]),
    "fp8rl_gemm_dgrad": (ST, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t, STREAM]),
    "fp8rl_gemm_wgrad": (ST, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t, STREAM]),
    "fp8rl_gemm_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, I64, I64, I64]),
    "fp8rl_gemm_workspace_bytes_ex": (ctypes.c_size_t, [ctypes.c_int, I64, I64, I64,
                                                        ctypes.POINTER(GemmOpts)]),
    "fp8rl_gemm_fwd_ex": (ST, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t,
                               ctypes.POINTER(GemmOpts), STREAM]),
    "fp8rl_gemm_dgrad_ex": (ST, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t,
                                 ctypes.POINTER(GemmOpts), STREAM]),
    "fp8rl_gemm_wgrad_ex": (ST, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t,
                                 ctypes.POINTER(GemmOpts), STREAM]),
    "fp8rl_linear_fwd": (ST, [P, I64, I64, I64, P, P, I64, P, P, P, P, ctypes.c_size_t, STREAM]),
    "fp8rl_gemm_fwd_decode_noalloc": (ST, [P, P, P, P, P, I64, I64, I64, STREAM]),
    "fp8rl_gemm_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "fp8rl_nvfp4_scale_bytes": (ctypes.c_size_t, [I64, I64]),
    "fp8rl_quantize_nvfp4": (ST, [P, I64, I64, I64, P, P, P, STREAM]),
    "fp8rl_gemm_nvfp4": (ST, [P, P, P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, STREAM]),
    "fp8rl_linear_nvfp4": (ST, [P, I64, I64, I64, P, P, P, I64, P, P, P, P, STREAM]),
    "fp8rl_debug_e4m3_encode": (ST, [P, P, I64, STREAM]),
    "fp8rl_debug_e2m1_encode": (ST, [P, P, I64, STREAM]),
    "fp8rl_debug_encode_check": (ST, [ctypes.c_uint32, ctypes.c_uint32, P, P, STREAM]),
    "fp8rl_debug_wait_timeout": (ST, [ctypes.c_uint64, STREAM]),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libfp8rl (declared signatures); raises if it was never built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libfp8rl.so is missing at {LIB_PATH}: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def check(status: int, where: str) -> None:
    if status != FP8RL_OK:
        raise Fp8rlError(status, where)
