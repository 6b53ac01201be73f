"""fp8rl_gemm_fwd_decode_noalloc: the decode-shaped forward GEMM for callers that cannot
give the library device memory (a C/C++ decode loop linking only this library, with no
allocator of its own, or a loop that must not allocate).  It runs on a scratch array
inside the library instead of a caller workspace.

Called here through the C ABI, twice in a row on each shape (the second call finds the
first call's leftovers in the shared scratch array).  Each call's output must be within
the GEMM tolerance the other tests use of the CPU oracle's unrounded result, and of the
allocating entry point (fp8rl_gemm_fwd_ex, split-K form, automatic splits).  Kept in a
file of its own, collected last, so that a failure here comes after every other test has
run.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth
from parity import bits16, gemm_tolerance_check, u8, f32

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _oracle_ref(oracle, qx, sx, qw, sw, M, N):
    """The oracle's result on every output of small problems, else on every row of a
    sample of 96 columns and every column of 4 rows (each element is independent)."""
    if M * N <= 1 << 20:
        return None, oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    rng = np.random.default_rng(M + N)
    cols = rng.choice(N, 96, replace=False)
    rows = rng.choice(M, min(4, M), replace=False)
    r1 = np.concatenate([np.repeat(np.arange(M), len(cols)), np.repeat(rows, N)])
    r2 = np.concatenate([np.tile(cols, M), np.tile(np.arange(N), len(rows))])
    return (r1, r2), oracle.gemm_sampled(u8(qx), f32(sx), u8(qw), f32(sw), "fwd", r1, r2)


@pytest.mark.parametrize("M,N,K", [(64, 3584, 3584), (256, 4608, 3584), (7, 1280, 1024),
                                   (256, 3584, 18944), (256, 28672, 4096)])
def test_noalloc_decode_matches_oracle_and_allocating_entry_point(fp8lib, oracle, M, N, K):
    lib = _abi.lib()
    x = synth.normal_bf16((M, K), 1.0, M + N, "cuda", outlier_channels=4, outlier_scale=30.0)
    w = synth.normal_bf16((N, K), 0.02, K + 1, "cuda")
    qx, sx = fp8lib.quantize_1x128(x)
    qw, sw, _ = fp8lib.quantize_128x128(w, transpose=False)
    idx, ref = _oracle_ref(oracle, qx, sx, qw, sw, M, N)
    y_alloc = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_SPLITK)
    ya = (bits16(y_alloc).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.fp8rl_gemm_fwd_decode_noalloc(_p(qx), _p(sx), _p(qw), _p(sw), _p(y), M, N, K,
                                               _stream())
        assert st == _abi.FP8RL_OK, _abi.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        yb = bits16(y)
        got = yb if idx is None else yb[idx[0], idx[1]]
        gemm_tolerance_check(got, ref, f"no-alloc decode {M}x{N}x{K} vs oracle, call {call}")
        gemm_tolerance_check(yb, ya, f"no-alloc decode {M}x{N}x{K} vs fp8rl_gemm_fwd_ex, call {call}")
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_noalloc_runs_every_decode_shape_and_rejects_large_m(fp8lib, oracle):
    lib = _abi.lib()
    cap = lib.fp8rl_gemm_noalloc_scratch_bytes()
    assert cap == 32 << 20
    # every 256-token decode problem of the 7B and 32B layers runs inside the array with
    # its automatic split; checked on 64 columns against the oracle
    for i, (N, K) in enumerate([(4608, 3584), (3584, 3584), (37888, 3584), (3584, 18944),
                                (7168, 5120), (5120, 5120), (55296, 5120), (5120, 27648)]):
        x = synth.normal_bf16((256, K), 1.0, 50 + i, "cuda")
        w = synth.normal_bf16((N, K), 0.015, 60 + i, "cuda")
        qx, sx = fp8lib.quantize_1x128(x)
        qw, sw, _ = fp8lib.quantize_128x128(w, transpose=False)
        y = torch.full((256, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.fp8rl_gemm_fwd_decode_noalloc(_p(qx), _p(sx), _p(qw), _p(sw), _p(y), 256, N, K, _stream())
        assert st == _abi.FP8RL_OK, (N, K, _abi.STATUS_NAMES.get(st, st))
        torch.cuda.synchronize()
        cols = np.random.default_rng(i).choice(N, 64, replace=False)
        r1 = np.repeat(np.arange(256), 64)
        r2 = np.tile(cols, 256)
        ref = oracle.gemm_sampled(u8(qx), f32(sx), u8(qw), f32(sw), "fwd", r1, r2)
        gemm_tolerance_check(bits16(y)[r1, r2], ref, f"no-alloc decode 256x{N}x{K}")
        del x, w, qx, sx, qw, sw, y
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")   # never read: rejected first
    st = lib.fp8rl_gemm_fwd_decode_noalloc(_p(t), _p(t), _p(t), _p(t), _p(t), 257, 128, 128, _stream())
    assert st == _abi.FP8RL_ERR_SHAPE
    assert fp8lib.check_status() == _abi.FP8RL_OK
