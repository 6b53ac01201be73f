"""GPU quantizers vs the CPU oracle: codes and scales bit-exact.

"Technical summary: Jet-RL", section "Quantization Scheme": activations 1x128, weights
128x128, WGrad operands 128x1 (emitted transposed).  Inputs are seeded synthetic BF16
generated on the GPU and copied to the host, so both sides see the same bytes.  Shapes span
several 128-wide groups/tiles, ragged M, strided rows, and the degenerate groups (all zero,
denormal amax, exact E4M3 rounding midpoints that exercise the exact-division fallback).
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import synth
from parity import assert_same_bits_f32, assert_same_u8, bits16, f32, u8

pytestmark = pytest.mark.gpu


def special_rows(M, K, device):
    """Rows built to hit the quantizer's edge cases (M >= 8)."""
    x = synth.normal_bf16((M, K), 1.0, 77, device).float()
    x[0] = 0.0                                       # all-zero groups
    x[1] = 0.0
    x[1, 0] = 2.0 ** -130                            # denormal amax -> saturation
    x[1, 1] = -(2.0 ** -131)
    x[2] = -0.0                                      # negative zeros
    # exact E4M3 midpoints after scaling by s = 2^3 (amax = 448 * 8)
    mids = torch.tensor([1.0625, 17.0, 432.0, 1.5 * 2 ** -9, 0.5 * 2 ** -9, 3.25, 5.5 * 2 ** -9],
                        device=device)
    row = torch.zeros(K, device=device)
    row[: mids.numel()] = mids * 8.0
    row[mids.numel():] = -mids.repeat(K // mids.numel() + 1)[: K - mids.numel()] * 8.0
    for g in range(K // 128):
        row[g * 128 + 100] = 448.0 * 8.0
    x[3] = row
    x[4] = row * 2.0 ** -20                          # same, tiny scale
    x[5] = 3.0e38 * torch.sign(x[5])                 # huge values
    x[6, ::3] = 0.0                                  # sparse row
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(1, 128), (7, 256), (128, 512), (300, 384), (1000, 1024)])
def test_quantize_1x128(fp8lib, oracle, M, K):
    x = synth.normal_bf16((M, K), 1.0, M * 31 + K, "cuda", outlier_channels=2, outlier_scale=30.0)
    if M >= 8:
        x = special_rows(M, K, "cuda")
    q, s = fp8lib.quantize_1x128(x)
    qr, sr = oracle.quantize_1x128(bits16(x))
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")


def test_quantize_1x128_strided_rows(fp8lib, oracle):
    base = synth.normal_bf16((200, 640), 2.0, 5, "cuda")
    x = base[:, 128:512]                            # ldx = 640 > K = 384
    q, s = fp8lib.quantize_1x128(x)
    qr, sr = oracle.quantize_1x128(bits16(x.contiguous()))
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")


@pytest.mark.parametrize("M,K", [(128, 128), (384, 640), (256, 1024)])
def test_quantize_dual(fp8lib, oracle, M, K):
    x = special_rows(M, K, "cuda")
    q, s, qT, sT = fp8lib.quantize_1x128(x, dual=True)
    xb = bits16(x)
    qr, sr = oracle.quantize_1x128(xb)
    qTr, sTr = oracle.quantize_128x1(xb)
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")
    assert_same_u8(u8(qT), qTr, "qT")
    assert_same_bits_f32(f32(sT), sTr, "sT")


def test_quantize_dual_tiny_columns(fp8lib, oracle):
    """128x1 groups whose scale is below 2^-68 (the exact-division fallback), one of them
    of BF16 denormals, and an all-zero column, beside ordinary columns of the same tiles."""
    M, K = 256, 512
    x = synth.normal_bf16((M, K), 1.0, 5, "cuda").float()
    x[128:256, 130] *= 2.0 ** -100
    x[128:256, 131] = 0.0
    x[0:128, 300:308] *= 2.0 ** -90
    x[0:128, 511] = 0.0
    x[17, 511] = 2.0 ** -133
    x[90, 511] = -(2.0 ** -132)
    x = x.to(torch.bfloat16)
    q, s, qT, sT = fp8lib.quantize_1x128(x, dual=True)
    xb = bits16(x)
    qr, sr = oracle.quantize_1x128(xb)
    qTr, sTr = oracle.quantize_128x1(xb)
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")
    assert_same_u8(u8(qT), qTr, "qT")
    assert_same_bits_f32(f32(sT), sTr, "sT")
    st = f32(sT)
    assert 0.0 < st[1, 130] < 2.0 ** -68 and st[1, 131] == 0.0 and 0.0 < st[0, 511] < 2.0 ** -68


@pytest.mark.parametrize("M,K", [(128, 256), (512, 384)])
def test_quantize_128x1(fp8lib, oracle, M, K):
    x = synth.normal_bf16((M, K), 1e-3, 11 + M, "cuda")
    qT, sT = fp8lib.quantize_128x1(x)
    qTr, sTr = oracle.quantize_128x1(bits16(x))
    assert_same_u8(u8(qT), qTr, "qT")
    assert_same_bits_f32(f32(sT), sTr, "sT")


@pytest.mark.parametrize("N,K,transpose", [(128, 128, True), (384, 512, True), (256, 384, False)])
def test_quantize_128x128(fp8lib, oracle, N, K, transpose):
    w = synth.normal_bf16((N, K), 0.02, N + K, "cuda")
    w[0, 0] = 0.5   # one large element per first block
    q, s, qT = fp8lib.quantize_128x128(w, transpose=transpose)
    qr, sr, qTr = oracle.quantize_128x128(bits16(w))
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")
    if transpose:
        assert_same_u8(u8(qT), qTr, "qT")
    else:
        assert qT is None


def test_quantize_128x128_strided_and_zero_block(fp8lib, oracle):
    base = synth.normal_bf16((256, 768), 0.02, 3, "cuda")
    base[:128, 256:384] = 0.0
    w = base[:, 256:640]
    q, s, qT = fp8lib.quantize_128x128(w)
    qr, sr, qTr = oracle.quantize_128x128(bits16(w.contiguous()))
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")
    assert_same_u8(u8(qT), qTr, "qT")
    assert f32(s)[0, 0] == 0.0


def test_quantize_128x128_tiny_blocks_in_a_long_sequence(fp8lib, oracle):
    """512 blocks over at most 304 persistent CTAs, so CTAs run a second block. Two blocks
    have amax small enough that their scale is below 2^-68 (the exact-division fallback),
    one of them with BF16 denormals."""
    N, K = 2048, 4096
    w = synth.normal_bf16((N, K), 0.02, 17, "cuda")
    w[3 * 128:4 * 128, 5 * 128:6 * 128] *= 2.0 ** -90           # amax ~2^-96: scale ~2^-105
    w[10 * 128:11 * 128, 20 * 128:21 * 128] = 0.0
    w[10 * 128 + 7, 20 * 128 + 9] = 2.0 ** -130                 # BF16 denormal, alone in its block
    w[10 * 128 + 100, 20 * 128 + 1] = -(2.0 ** -131)
    q, s, qT = fp8lib.quantize_128x128(w)
    qr, sr, qTr = oracle.quantize_128x128(bits16(w))
    assert_same_u8(u8(q), qr, "q")
    assert_same_bits_f32(f32(s), sr, "s")
    assert_same_u8(u8(qT), qTr, "qT")
    assert 0.0 < f32(s)[3, 5] < 2.0 ** -68 and 0.0 < f32(s)[10, 20] < 2.0 ** -68


def test_device_encoder_exhaustive(fp8lib, oracle):
    """The device E4M3 conversion equals the oracle's encoder on every finite binary32."""
    chunk = 1 << 28
    for c in range(16):
        start = c * chunk
        idx = torch.arange(chunk, dtype=torch.int64, device="cuda") + start
        v = (idx & 0xFFFFFFFF).to(torch.int64)
        v = torch.where(v >= 2 ** 31, v - 2 ** 32, v).to(torch.int32).view(torch.float32)
        got = u8(fp8lib.debug_e4m3_encode(v))
        ref = oracle.e4m3_encode_bits_range(start, chunk)
        vals = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        fin = np.isfinite(vals)
        bad = (got != ref) & fin
        assert not bad.any(), f"chunk {c}: {int(bad.sum())} differ, e.g. bits {np.nonzero(bad)[0][0] + start:#x}"
        del idx, v


def test_division_free_encode_is_exact_for_every_bf16_pair(fp8lib):
    """The quantizers form x/s from RN(1/s) with one correction step instead of dividing.
    Their inputs are BF16 values, so the whole domain is finite: every positive finite BF16
    group maximum against every BF16 x with |x| <= amax (both signs and zeros) must give the
    same E4M3 code as IEEE division."""
    mismatches, first = fp8lib.debug_encode_check(1, 0x7F80)
    assert mismatches == 0, f"{mismatches} mismatches, first amax/x bits {first:#010x}"
