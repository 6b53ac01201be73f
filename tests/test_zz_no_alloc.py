"""fp8rl_gemm_fwd_decode_noalloc: the decode-shaped forward GEMM for callers that cannot
give the library device memory (a C/C++ decode loop linking only this library, with no
allocator of its own, or a loop that must not allocate).  It runs on a scratch array
inside the library instead of a caller workspace.

Called here through the C ABI; its output must match the allocating entry point
(fp8rl_gemm_fwd_ex, split-K form, automatic splits) within the GEMM tolerance the other
tests use, on two calls in a row (the second call finds the first call's leftovers in the
shared scratch array).  Kept in a file of its own, collected last, so that a failure here
comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth
from parity import bits16, gemm_tolerance_check

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("M,N,K", [(64, 3584, 3584), (256, 4608, 3584), (7, 1280, 1024),
                                   (256, 3584, 18944), (256, 28672, 4096)])
def test_noalloc_decode_matches_allocating_entry_point(fp8lib, M, N, K):
    lib = _abi.lib()
    x = synth.normal_bf16((M, K), 1.0, M + N, "cuda")
    w = synth.normal_bf16((N, K), 0.02, K + 1, "cuda")
    qx, sx = fp8lib.quantize_1x128(x)
    qw, sw, _ = fp8lib.quantize_128x128(w, transpose=False)
    y_ref = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_SPLITK)
    ref = (bits16(y_ref).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.fp8rl_gemm_fwd_decode_noalloc(_p(qx), _p(sx), _p(qw), _p(sw), _p(y), M, N, K,
                                               _stream())
        assert st == _abi.FP8RL_OK, _abi.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        gemm_tolerance_check(bits16(y), ref, f"no-alloc decode {M}x{N}x{K}, call {call}")
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_noalloc_runs_every_decode_shape_and_rejects_large_m(fp8lib):
    lib = _abi.lib()
    cap = lib.fp8rl_gemm_noalloc_scratch_bytes()
    assert cap == 32 << 20
    # every 256-token decode problem of the 7B and 32B layers runs inside the array: with
    # the automatic split where its partial sums fit, else with a smaller one (zero
    # operands, so the product is exactly zero)
    for N, K in [(4608, 3584), (3584, 3584), (37888, 3584), (3584, 18944), (7168, 5120),
                 (5120, 5120), (55296, 5120), (5120, 27648)]:
        qx = torch.zeros((256, K), dtype=torch.uint8, device="cuda")
        sx = torch.zeros((K // 128, 256), dtype=torch.float32, device="cuda")
        qw = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
        sw = torch.zeros((N // 128, K // 128), dtype=torch.float32, device="cuda")
        y = torch.full((256, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.fp8rl_gemm_fwd_decode_noalloc(_p(qx), _p(sx), _p(qw), _p(sw), _p(y), 256, N, K, _stream())
        assert st == _abi.FP8RL_OK, (N, K, _abi.STATUS_NAMES.get(st, st))
        torch.cuda.synchronize()
        assert bool((y == 0).all()), (N, K)
        del qx, sx, qw, sw, y
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")   # never read: rejected first
    st = lib.fp8rl_gemm_fwd_decode_noalloc(_p(t), _p(t), _p(t), _p(t), _p(t), 257, 128, 128, _stream())
    assert st == _abi.FP8RL_ERR_SHAPE
    assert fp8lib.check_status() == _abi.FP8RL_OK
