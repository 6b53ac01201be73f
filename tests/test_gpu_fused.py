"""Fused RMSNorm -> quantize and SiLU-mul -> quantize on the GPU vs the CPU oracle.

"Technical summary: Jet-RL", section "Implementation" (fused activation / RMSNorm kernels
feeding quantization) and section "Quantization Scheme" (saved activations in FP8, 1x128
and the transposed 128x1 copy for WGrad).

RMSNorm: the device sums squares in a different order than the oracle's binary64 loop, so
rstd may differ in the last place for rare rows.  Check: rstd bit-equal or within 1 ulp;
then every code and scale bit-exact against the oracle fed the device's rstd.  (With an
rstd buffer the device computes rstd in a separate kernel first; without one, inside a
cluster of CTAs per panel: both are covered.)

SiLU-mul: the device evaluates silu(g)*u in binary32 (exp and a fast reciprocal), the
oracle in binary64; they can round h to different BF16 neighbours only where the binary64
value lies within 2^-16 of a BF16 midpoint.  Groups without such elements must be
bit-exact; groups with them must equal the oracle's quantization of one of the choices.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import synth
from parity import assert_same_bits_f32, assert_same_u8, bits16, f32, silu_group_matches, u8

pytestmark = pytest.mark.gpu


def check_rmsnorm(fp8lib, oracle, x, gamma, eps, dual):
    q, s, qT, sT, rstd = fp8lib.rmsnorm_quant(x, gamma, eps, dual=dual)
    xb, gb = bits16(x), bits16(gamma)
    _, _, _, _, r_ref, _ = oracle.rmsnorm_quant(xb, gb, eps)
    r_gpu = f32(rstd)
    diff = r_gpu.view(np.int32).astype(np.int64) - r_ref.view(np.int32).astype(np.int64)
    assert np.all(np.abs(diff) <= 1), f"rstd off by more than 1 ulp in {int((np.abs(diff) > 1).sum())} rows"
    qr, sr, qTr, sTr, _, _ = oracle.rmsnorm_quant(xb, gb, eps, rstd_in=r_gpu)
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")
    if dual:
        assert_same_u8(u8(qT), qTr, "qT")
        assert_same_bits_f32(f32(sT), sTr, "sT")
    return int((diff != 0).sum())


# 6272 = 49 x 128 K-blocks: the cluster form splits a panel 7 ways
@pytest.mark.parametrize("M,K", [(128, 128), (256, 640), (384, 1024), (128, 4096), (256, 5120),
                                 (128, 6144), (256, 6272)])
def test_rmsnorm_quant_dual(fp8lib, oracle, M, K):
    x = synth.normal_bf16((M, K), 1.0, M + K, "cuda", outlier_channels=max(1, K // 1000),
                          outlier_scale=30.0)
    x[3] = 0.0                       # zero row
    x[5] = 2.5                       # constant row
    gamma = synth.normal_bf16((K,), 0.1, 9, "cuda").float().add_(1.0).to(torch.bfloat16)
    check_rmsnorm(fp8lib, oracle, x, gamma, 1e-5, dual=True)


@pytest.mark.parametrize("M,K", [(1, 256), (100, 384), (1000, 1024)])
def test_rmsnorm_quant_rows_only(fp8lib, oracle, M, K):
    x = synth.normal_bf16((M, K), 1.0, 3 * M + K, "cuda")
    gamma = torch.ones(K, dtype=torch.bfloat16, device="cuda")
    check_rmsnorm(fp8lib, oracle, x, gamma, 1e-6, dual=False)


@pytest.mark.parametrize("M,K", [(256, 640), (384, 1024), (128, 4096), (256, 6272)])
def test_rmsnorm_quant_without_rstd_buffer(fp8lib, M, K):
    """Without an rstd buffer the library computes rstd inside a cluster of CTAs per panel
    (it allocates nothing).  Its codes and scales equal those of the path that writes rstd
    first, on these seeded inputs (the two sum the squares in different orders, which
    could move rstd by one ulp only for a row whose mean square sits on a rounding
    boundary of binary32)."""
    import ctypes

    from block_scaled_fp8_x1_gb300 import _abi
    x = synth.normal_bf16((M, K), 1.0, 7 * M + K, "cuda", outlier_channels=2, outlier_scale=30.0)
    gamma = synth.normal_bf16((K,), 0.1, 4, "cuda").float().add_(1.0).to(torch.bfloat16)
    q1, s1, qT1, sT1, _ = fp8lib.rmsnorm_quant(x, gamma, 1e-5, dual=True)
    q2, s2 = torch.empty_like(q1), torch.empty_like(s1)
    qT2, sT2 = torch.empty_like(qT1), torch.empty_like(sT1)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = _abi.lib().fp8rl_rmsnorm_quant(p(x), p(gamma), ctypes.c_float(1e-5), M, K, p(q2), p(s2), p(qT2),
                                        p(sT2), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _abi.FP8RL_OK
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(qT1, qT2)
    assert torch.equal(s1.view(torch.int32), s2.view(torch.int32))
    assert torch.equal(sT1.view(torch.int32), sT2.view(torch.int32))
    assert fp8lib.check_status() == _abi.FP8RL_OK


def check_silu(fp8lib, oracle, gu, dual):
    q, s, qT, sT = fp8lib.silu_mul_quant(gu, dual=dual)
    h, alt, nflag = oracle.silu_mul(bits16(gu))
    qr, sr = oracle.quantize_1x128(h)
    qg, sg = u8(q), f32(s)
    M, I = h.shape
    n_inexact = 0
    for m in range(M):
        for b in range(I // 128):
            sl = slice(b * 128, (b + 1) * 128)
            if np.array_equal(qg[m, sl], qr[m, sl]) and sg[b, m].view(np.uint32) == sr[b, m].view(np.uint32):
                continue
            n_inexact += 1
            assert silu_group_matches(oracle, qg[m, sl], sg[b, m], h[m, sl], alt[m, sl]), (m, b)
    if dual:
        qTr, sTr = oracle.quantize_128x1(h)
        qTg, sTg = u8(qT), f32(sT)
        for i in range(I):
            for b in range(M // 128):
                sl = slice(b * 128, (b + 1) * 128)
                if np.array_equal(qTg[i, sl], qTr[i, sl]) and sTg[b, i].view(np.uint32) == sTr[b, i].view(np.uint32):
                    continue
                n_inexact += 1
                assert silu_group_matches(oracle, qTg[i, sl], sTg[b, i], h[sl, i], alt[sl, i]), (i, b)
    return n_inexact, nflag


@pytest.mark.parametrize("M,I", [(128, 128), (256, 384), (384, 1024)])
def test_silu_mul_quant_dual(fp8lib, oracle, M, I):
    gu = synth.normal_bf16((M, 2 * I), 2.0, M * 7 + I, "cuda")
    gu[0, :I] = 0.0                  # silu(0) = 0 -> zero group
    gu[1, :I] = 40.0                 # silu(g) ~ g
    gu[2, I:] = 0.0                  # u = 0
    n_inexact, nflag = check_silu(fp8lib, oracle, gu, dual=True)
    assert n_inexact <= nflag * 2


def test_silu_mul_quant_rows_only_ragged(fp8lib, oracle):
    gu = synth.normal_bf16((77, 2 * 256), 1.5, 4, "cuda")
    check_silu(fp8lib, oracle, gu, dual=False)
