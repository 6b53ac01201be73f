"""The backward operators either side of the gradient quantizer, on the GPU vs the oracle.

"Technical summary: Jet-RL", section "Quantization Scheme": gradients between operators
stay BF16 and DGrad / WGrad run on gradients quantized 1x128 and 128x1.

SiLU-mul backward -> quantize: the device evaluates dg, du in binary32 (exp and a fast
reciprocal), the oracle in binary64; they can round to different BF16 neighbours only where
the oracle flags an element as near a BF16 midpoint (relative to the size of its terms).
Groups without such elements must be bit-exact in codes and scales; groups with them must
equal the oracle's quantization of one of the choices.

RMSNorm backward: dx within one BF16 rounding of the oracle's binary64 value plus binary32
evaluation error, |dx - ref| <= 2^-8 (|r gamma dy| + |r^3 x S / K|); dgamma within
2^-12 sum_m |dy x r| (binary32 sums of up to 16384 rows, compensated); repeat calls give
identical bits.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth
from parity import bits16, f32, silu_group_matches, u8

pytestmark = pytest.mark.gpu


def check_silu_bwd(fp8lib, oracle, gu, dh, dual):
    q, s, qT, sT = fp8lib.silu_mul_bwd_quant(gu, dh, dual=dual)
    dgu, alt, nflag = oracle.silu_mul_bwd(bits16(gu), bits16(dh))
    qr, sr = oracle.quantize_1x128(dgu)
    qg, sg = u8(q), f32(s)
    M, C = dgu.shape
    n_inexact = 0
    # groups that differ from the oracle's bytes must match one of its flagged choices
    same = (qg.reshape(M, C // 128, 128) == qr.reshape(M, C // 128, 128)).all(axis=2) & (
        sg.T.view(np.uint32) == sr.T.view(np.uint32))
    for m, b in np.argwhere(~same):
        sl = slice(b * 128, (b + 1) * 128)
        n_inexact += 1
        assert silu_group_matches(oracle, qg[m, sl], sg[b, m], dgu[m, sl], alt[m, sl]), (m, b)
    if dual:
        qTr, sTr = oracle.quantize_128x1(dgu)
        qTg, sTg = u8(qT), f32(sT)
        same = (qTg.reshape(C, M // 128, 128) == qTr.reshape(C, M // 128, 128)).all(axis=2) & (
            sTg.T.view(np.uint32) == sTr.T.view(np.uint32))
        for c, b in np.argwhere(~same):
            sl = slice(b * 128, (b + 1) * 128)
            n_inexact += 1
            assert silu_group_matches(oracle, qTg[c, sl], sTg[b, c], dgu[sl, c], alt[sl, c]), (c, b)
    return n_inexact, nflag


@pytest.mark.parametrize("M,I", [(128, 128), (256, 384), (384, 1024)])
def test_silu_mul_bwd_quant_dual(fp8lib, oracle, M, I):
    gu = synth.normal_bf16((M, 2 * I), 2.0, 5 * M + I, "cuda")
    dh = synth.normal_bf16((M, I), 1e-3, 3 * M + I, "cuda")
    gu[0, :I] = 0.0                  # g = 0: dg = dh*u/2, du = 0 (a zero group of du)
    gu[1, :I] = 30.0                 # saturated sigmoid
    dh[2] = 0.0                      # zero gradient row
    gu[3, :I] = -1.28125             # next to the root of silu' (dg cancels)
    n_inexact, nflag = check_silu_bwd(fp8lib, oracle, gu, dh, dual=True)
    assert n_inexact <= 2 * nflag
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_silu_mul_bwd_quant_dual_many_items_per_cta(fp8lib, oracle):
    """1024 source blocks over at most 304 persistent CTAs: each CTA runs several items, so
    the next item's tiles are requested in two parts while the codes of the current one
    are staged in its gate tile."""
    M, I = 4096, 4096
    gu = synth.normal_bf16((M, 2 * I), 2.0, 17, "cuda")
    dh = synth.normal_bf16((M, I), 1e-3, 18, "cuda")
    n_inexact, nflag = check_silu_bwd(fp8lib, oracle, gu, dh, dual=True)
    assert n_inexact <= 2 * nflag
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_silu_mul_bwd_quant_rows_only_ragged(fp8lib, oracle):
    gu = synth.normal_bf16((77, 2 * 256), 1.5, 8, "cuda")
    dh = synth.normal_bf16((77, 256), 1e-2, 9, "cuda")
    check_silu_bwd(fp8lib, oracle, gu, dh, dual=False)


@pytest.mark.parametrize("M,K", [(128, 128), (300, 640), (1000, 4096), (257, 5120), (64, 8192)])
def test_rmsnorm_bwd(fp8lib, oracle, M, K):
    x = synth.normal_bf16((M, K), 1.0, M + K, "cuda", outlier_channels=max(1, K // 1000), outlier_scale=30.0)
    x[1] = 0.0                       # zero row
    x[2] = 1.5                       # constant row
    gamma = synth.normal_bf16((K,), 0.1, 6, "cuda").float().add_(1.0).to(torch.bfloat16)
    dy = synth.normal_bf16((M, K), 1e-3, 2 * M + K, "cuda")
    _, _, _, _, rstd = fp8lib.rmsnorm_quant(x, gamma, 1e-5, dual=False)
    dx, dgamma = fp8lib.rmsnorm_bwd(x, gamma, rstd, dy)
    xr, gr, dyr, rr = bits16(x), bits16(gamma), bits16(dy), f32(rstd)
    dx_ref, mag, dg_ref = oracle.rmsnorm_bwd(xr, gr, rr, dyr)
    got = (bits16(dx).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = (dx_ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # ref is the BF16 rounding of the binary64 value: one more BF16 rounding allowed
    bad = np.abs(got - ref) > 2.0 ** -8 * mag + 2.0 ** -8 * np.abs(ref) + 1e-30
    assert not bad.any(), f"{int(bad.sum())} dx outside the bound, first at {np.argwhere(bad)[0]}"
    def b2f(b):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    absum = np.sum(np.abs(b2f(dyr) * b2f(xr) * rr.astype(np.float64)[:, None]), axis=0)
    dg = f32(dgamma).astype(np.float64)
    assert np.all(np.abs(dg - dg_ref) <= 2.0 ** -12 * absum + 1e-30)
    dx2, dgamma2 = fp8lib.rmsnorm_bwd(x, gamma, rstd, dy)
    assert torch.equal(dx.view(torch.int16), dx2.view(torch.int16))
    assert torch.equal(dgamma.view(torch.int32), dgamma2.view(torch.int32))
    dx3, none = fp8lib.rmsnorm_bwd(x, gamma, rstd, dy, with_dgamma=False)
    assert none is None and torch.equal(dx.view(torch.int16), dx3.view(torch.int16))
    assert fp8lib.check_status() == _abi.FP8RL_OK


@pytest.mark.parametrize("M,K", [(128, 128), (256, 640), (1024, 384)])
def test_requantize_128x1_matches_oracle(fp8lib, oracle, M, K):
    x = synth.normal_bf16((M, K), 1.0, M + 3 * K, "cuda", outlier_channels=2, outlier_scale=30.0)
    x[:, 5] = 0.0                    # a zero column: zero groups after the round trip
    q, s = fp8lib.quantize_1x128(x)
    qT, sT = fp8lib.requantize_128x1(q, s)
    qTr, sTr = oracle.requant_128x1(u8(q), f32(s))
    assert np.array_equal(u8(qT), qTr)
    assert np.array_equal(f32(sT).view(np.uint32), sTr.view(np.uint32))
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_wgrad_from_saved_fp8_extra_error(fp8lib, oracle):
    """The memory-saving WGrad (activation operand rebuilt from its saved 1x128 FP8) against
    the WGrad from the BF16 activation: both against the exact dW = dY^T X of the BF16
    inputs (binary64).  The extra error is the 1x128 rounding the saved form starts from:
    measured here, and bounded at three times the direct path's relative error."""
    M, N, K = 1024, 512, 768
    dy = synth.normal_bf16((M, N), 1e-3, 91, "cuda")
    x = synth.normal_bf16((M, K), 1.0, 92, "cuda", outlier_channels=2, outlier_scale=30.0)
    qdyT, sdyT = fp8lib.quantize_128x1(dy)
    qxT, sxT = fp8lib.quantize_128x1(x)
    q1, s1 = fp8lib.quantize_1x128(x)
    qxT2, sxT2 = fp8lib.requantize_128x1(q1, s1)
    dw_direct = fp8lib.gemm_wgrad(qdyT, sdyT, qxT, sxT)
    dw_saved = fp8lib.gemm_wgrad(qdyT, sdyT, qxT2, sxT2)
    b2f = lambda t: (bits16(t).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = b2f(dy).T @ b2f(x)
    norm = np.linalg.norm(exact)
    e_direct = np.linalg.norm(b2f(dw_direct) - exact) / norm
    e_saved = np.linalg.norm(b2f(dw_saved) - exact) / norm
    print(f"WGrad relative Frobenius error: from BF16 {e_direct:.3e}, from saved FP8 {e_saved:.3e}")
    assert e_direct < 0.05 and e_saved <= 3.0 * e_direct
    # and the saved-form WGrad is the oracle's GEMM of its own operands
    ref = oracle.gemm(u8(qdyT), f32(sdyT), u8(qxT2), f32(sxT2), "wgrad")
    from parity import gemm_tolerance_check
    gemm_tolerance_check(bits16(dw_saved), ref, "WGrad from saved FP8")
