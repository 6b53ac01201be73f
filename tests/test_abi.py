"""The C ABI library builds, loads and exports every entry point include/fp8rl.h declares;
host-side argument checks answer without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8rl.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8rl_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def abi():
    from block_scaled_fp8_x1_gb300 import build_library
    from block_scaled_fp8_x1_gb300 import _abi
    build_library()
    return _abi


def test_every_declared_symbol_is_exported(abi):
    L = abi.lib()
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
        assert n in abi.SIGNATURES, f"binding lacks {n}"


def test_binding_names_are_declared(abi):
    assert set(abi.SIGNATURES) == set(declared_functions())


def test_status_strings(abi):
    L = abi.lib()
    for code, name in abi.STATUS_NAMES.items():
        assert L.fp8rl_status_string(code).decode() == name


def test_host_side_validation_without_gpu(abi):
    L = abi.lib()
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails first
    odd = ctypes.c_void_p(0x10004)
    null = None
    # shape rules
    assert L.fp8rl_quantize_1x128(fake, 4, 100, 100, fake, fake, null, null, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_quantize_1x128(fake, 100, 128, 128, fake, fake, fake, fake, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_quantize_128x1(fake, 100, 128, 128, fake, fake, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_quantize_128x128(fake, 100, 128, 128, fake, fake, null, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_silu_mul_quant(fake, 4, 100, fake, fake, null, null, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_gemm_fwd(fake, fake, fake, fake, fake, 4, 100, 128, null, 0, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_gemm_wgrad(fake, fake, fake, fake, fake, 100, 128, 128, null, 0, null) == abi.FP8RL_ERR_SHAPE
    # bad arguments
    assert L.fp8rl_quantize_1x128(fake, -1, 128, 128, fake, fake, null, null, null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_quantize_1x128(fake, 4, 128, 64, fake, fake, null, null, null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_quantize_1x128(fake, 128, 128, 128, fake, fake, fake, null, null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_quantize_1x128(null, 4, 128, 128, fake, fake, null, null, null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_rmsnorm_quant(fake, fake, ctypes.c_float(-1.0), 4, 128, fake, fake, null, null, null, null) == abi.FP8RL_ERR_INVALID_ARG
    opts = abi.GemmOpts(7, 0, 0)
    assert L.fp8rl_gemm_fwd_ex(fake, fake, fake, fake, fake, 4, 128, 128, null, 0, ctypes.byref(opts), null) == abi.FP8RL_ERR_INVALID_ARG
    # DGrad / WGrad take AUTO, TILED or PAIR; the split-K form is forward-only
    splitk = abi.GemmOpts(abi.FP8RL_VARIANT_SPLITK, 0, 0)
    assert L.fp8rl_gemm_dgrad_ex(fake, fake, fake, fake, fake, 4, 128, 128, null, 0, ctypes.byref(splitk), null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_gemm_wgrad_ex(fake, fake, fake, fake, fake, 128, 128, 128, null, 0, ctypes.byref(opts), null) == abi.FP8RL_ERR_INVALID_ARG
    # alignment (16 bytes for every device pointer)
    assert L.fp8rl_quantize_1x128(odd, 4, 128, 128, fake, fake, null, null, null) == abi.FP8RL_ERR_ALIGN
    assert L.fp8rl_quantize_1x128(fake, 4, 128, 132, fake, fake, null, null, null) == abi.FP8RL_ERR_ALIGN
    assert L.fp8rl_gemm_dgrad(fake, fake, odd, fake, fake, 4, 128, 128, null, 0, null) == abi.FP8RL_ERR_ALIGN
    # empty problems are no-ops
    assert L.fp8rl_quantize_1x128(null, 0, 128, 128, null, null, null, null, null) == abi.FP8RL_OK
    assert L.fp8rl_gemm_fwd(null, null, null, null, null, 0, 128, 128, null, 0, null) == abi.FP8RL_OK
    assert L.fp8rl_gemm_dgrad(null, null, null, null, null, 0, 128, 128, null, 0, null) == abi.FP8RL_OK


def test_workspace_sizes(abi):
    L = abi.lib()
    # decode form (M <= 256) splitting the reduction needs its partial sums; tiled none
    # the automatic decode form for up to 64 tokens (128 for N <= 8192) reduces inside a
    # cluster: no workspace; the split-K form (otherwise up to 256 tokens) keeps its partial
    # sums in one
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_FWD, 64, 37888, 3584) == 0
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_FWD, 128, 3584, 3584) == 0
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_FWD, 128, 8320, 3584) > 0
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_FWD, 256, 3584, 3584) > 0
    # 256 tokens against a wide weight: the paired form, no workspace
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_FWD, 256, 37888, 3584) == 0
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_FWD, 8192, 3584, 3584) == 0
    assert L.fp8rl_gemm_workspace_bytes(abi.FP8RL_OP_WGRAD, 8192, 3584, 3584) == 0
    opts = abi.GemmOpts(abi.FP8RL_VARIANT_SPLITK, 4, 0)
    need = L.fp8rl_gemm_workspace_bytes_ex(abi.FP8RL_OP_FWD, 256, 3584, 3584, ctypes.byref(opts))
    assert need == 28 * 4 * 256 * 128 * 4
    one = abi.GemmOpts(abi.FP8RL_VARIANT_SPLITK, 1, 0)
    assert L.fp8rl_gemm_workspace_bytes_ex(abi.FP8RL_OP_FWD, 256, 3584, 3584, ctypes.byref(one)) == 0


def test_nvfp4_host_rules(abi):
    L = abi.lib()
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    null = None
    # scale-factor bytes: ceil(R/128) row groups x K/256 K-blocks x 2 KB
    assert L.fp8rl_nvfp4_scale_bytes(1, 256) == 2048
    assert L.fp8rl_nvfp4_scale_bytes(129, 3584) == 2 * 14 * 2048
    assert L.fp8rl_nvfp4_scale_bytes(37888, 3584) == 296 * 14 * 2048
    assert L.fp8rl_nvfp4_scale_bytes(64, 384) == 0 and L.fp8rl_nvfp4_scale_bytes(0, 256) == 0
    # K must be a multiple of 256, N of 128, M at most 256
    assert L.fp8rl_quantize_nvfp4(fake, 4, 384, 384, fake, fake, fake, null) == abi.FP8RL_ERR_SHAPE
    args = [fake] * 7
    assert L.fp8rl_gemm_nvfp4(*args, 4, 128, 384, 128, 0, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_gemm_nvfp4(*args, 4, 200, 256, 200, 0, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_gemm_nvfp4(*args, 257, 128, 256, 128, 0, null) == abi.FP8RL_ERR_SHAPE
    assert L.fp8rl_gemm_nvfp4(*args, 4, 128, 256, 64, 0, null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_gemm_nvfp4(*args, 4, 128, 256, 128, -1, null) == abi.FP8RL_ERR_INVALID_ARG
    assert L.fp8rl_linear_nvfp4(fake, 300, 256, 256, fake, fake, fake, 128, fake, fake, fake, fake, null) == abi.FP8RL_ERR_SHAPE
    # alignment and missing pointers
    assert L.fp8rl_quantize_nvfp4(odd, 4, 256, 256, fake, fake, fake, null) == abi.FP8RL_ERR_ALIGN
    assert L.fp8rl_quantize_nvfp4(fake, 4, 256, 260, fake, fake, fake, null) == abi.FP8RL_ERR_ALIGN
    assert L.fp8rl_gemm_nvfp4(fake, fake, fake, odd, fake, fake, fake, 4, 128, 256, 128, 0, null) == abi.FP8RL_ERR_ALIGN
    assert L.fp8rl_gemm_nvfp4(fake, fake, fake, fake, fake, fake, fake, 4, 128, 256, 132, 0, null) == abi.FP8RL_ERR_ALIGN
    assert L.fp8rl_quantize_nvfp4(fake, 4, 256, 256, fake, null, fake, null) == abi.FP8RL_ERR_INVALID_ARG
    # empty problems are no-ops
    assert L.fp8rl_quantize_nvfp4(null, 0, 256, 256, null, null, null, null) == abi.FP8RL_OK
    assert L.fp8rl_gemm_nvfp4(null, null, null, null, null, null, null, 0, 128, 256, 128, 0, null) == abi.FP8RL_OK
