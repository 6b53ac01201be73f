"""NVFP4 rollout path on the GPU vs the CPU oracle.

"QeRL" (chatpaper.ai), abstract: rollout runs with NVFP4-quantized weights.  The quantizer
must give the oracle's codes, block scales and row scales bit for bit (the block scales
read back from the tensor core's atom layout by the header's formula); the FP4 GEMM must
satisfy |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref) against the oracle's binary64 sum
on the same operands, and give the exact result where the FP32 accumulation is exact.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import synth
from parity import assert_same_bits_f32, assert_same_u8, bits16, f32, gemm_tolerance_check, u8

pytestmark = pytest.mark.gpu


def sf_rows(sf: torch.Tensor, R: int, K: int):
    """The atom layout (512-byte atoms of 128 rows x 4 scales, row r's scale j of the atom
    at byte 16 (r % 32) + 4 ((r % 128) / 32) + j) -> ([R, K/16], the padding rows)."""
    rp = (R + 127) // 128 * 128
    a = u8(sf).reshape(rp // 128, K // 64, 32, 4, 4)      # [rg][ka][r % 32][(r % 128) / 32][j]
    rows = a.transpose(0, 3, 2, 1, 4).reshape(rp, K // 16)
    return rows[:R], rows[R:]


def check_quant(fp8lib, oracle, x):
    R, K = x.shape
    q, sf, g = fp8lib.quantize_nvfp4(x)
    qr, sfr, gr = oracle.quantize_nvfp4(bits16(x.contiguous()))
    assert_same_u8(u8(q), qr, "q")
    rows, pad = sf_rows(sf, R, K)
    assert_same_u8(rows, sfr, "sf")
    assert not pad.any(), "padding rows of sf must be zero"
    assert_same_bits_f32(f32(g), gr, "g")
    return q, sf, g, qr, sfr, gr


def special_rows(R, K):
    x = synth.normal_bf16((R, K), 1.0, R + K, "cuda", outlier_channels=max(1, K // 500),
                          outlier_scale=30.0).float()
    x[0] = 0.0                                           # all-zero row
    x[1] = 0.0
    x[1, 3] = 2.0 ** -130                                # denormal maximum
    x[1, 200] = -(2.0 ** -133)
    x[2] = -0.0
    x[3, 17] = 1.0e4                                     # one outlier: tiny blocks flush to 0
    x[4] = 3.0e38 * torch.sign(x[4])                     # huge values
    x[5, ::3] = 0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("R,K", [(1, 256), (7, 512), (128, 256), (300, 768), (1000, 3584)])
def test_quantize_nvfp4(fp8lib, oracle, R, K):
    x = special_rows(R, K) if R >= 8 else synth.normal_bf16((R, K), 0.5, K, "cuda")
    check_quant(fp8lib, oracle, x)


def test_quantize_nvfp4_strided_rows(fp8lib, oracle):
    base = synth.normal_bf16((200, 1280), 0.02, 3, "cuda")
    x = base[:, 256:1024]                                  # ldx = 1280 > K = 768
    q, sf, g = fp8lib.quantize_nvfp4(x)
    qr, sfr, gr = oracle.quantize_nvfp4(bits16(x.contiguous()))
    assert_same_u8(u8(q), qr, "q")
    assert_same_u8(sf_rows(sf, 200, 768)[0], sfr, "sf")
    assert_same_bits_f32(f32(g), gr, "g")


def test_device_e2m1_encoder_exhaustive(fp8lib, oracle):
    """The device E2M1 conversion equals the oracle's encoder on every finite binary32."""
    chunk = 1 << 28
    for c in range(16):
        start = c * chunk
        idx = torch.arange(chunk, dtype=torch.int64, device="cuda") + start
        v = torch.where(idx >= 2 ** 31, idx - 2 ** 32, idx).to(torch.int32).view(torch.float32)
        got = u8(fp8lib.debug_e2m1_encode(v))
        ref = oracle.e2m1_encode_bits_range(start, chunk)
        vals = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        bad = (got != ref) & np.isfinite(vals)
        assert not bad.any(), f"chunk {c}: {int(bad.sum())} differ, e.g. bits {np.nonzero(bad)[0][0] + start:#x}"
        del idx, v


def operands(fp8lib, oracle, M, N, K, seed):
    x = synth.normal_bf16((M, K), 1.0, seed, "cuda", outlier_channels=max(1, K // 1000), outlier_scale=30.0)
    w = synth.normal_bf16((N, K), 0.02, seed + 1, "cuda")
    qx, sfx, gx, qxr, sfxr, gxr = check_quant(fp8lib, oracle, x)
    qw, sfw, gw, qwr, sfwr, gwr = check_quant(fp8lib, oracle, w)
    return (qx, sfx, gx, qw, sfw, gw), (qxr, sfxr, gxr, qwr, sfwr, gwr), x


# token counts around every padding class (32/64/128/256), cluster sizes from one CTA to
# one K-block per CTA
@pytest.mark.parametrize("M", [1, 5, 31, 32, 33, 64, 100, 128, 129, 200, 256])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_gemm_nvfp4(fp8lib, oracle, M, splits):
    N, K = 1280, 2048
    dev, ref, _ = operands(fp8lib, oracle, M, N, K, 11 * M + splits)
    y = fp8lib.gemm_nvfp4(*dev, splits=splits)
    y_ref = oracle.gemm_nvfp4(*ref)
    gemm_tolerance_check(bits16(y), y_ref, f"nvfp4 M={M} splits={splits}")
    y2 = fp8lib.gemm_nvfp4(*dev, splits=splits)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("splits", [1, 4])
def test_gemm_nvfp4_strided_output(fp8lib, oracle, splits):
    """y written into columns 128 .. 128 + N of a wider buffer (ldy > N); the columns
    around it stay untouched."""
    M, N, K = 100, 768, 1024
    dev, ref, _ = operands(fp8lib, oracle, M, N, K, 91 + splits)
    big = torch.full((M, N + 256), -7.0, dtype=torch.bfloat16, device="cuda")
    view = big[:, 128:128 + N]
    fp8lib.gemm_nvfp4(*dev, splits=splits, out=view)
    gemm_tolerance_check(bits16(view), oracle.gemm_nvfp4(*ref), f"nvfp4 ldy splits={splits}")
    assert torch.all(big[:, :128] == -7.0) and torch.all(big[:, 128 + N:] == -7.0)


def test_gemm_nvfp4_exact(fp8lib, oracle):
    """Operands whose FP32 accumulation is exact: every block holds a +-6 element and has
    scale 224 or 448, the row scales are powers of two, so each product is 49 * 2^k times
    an integer below 2^8 and every partial sum of K = 512 terms is an integer multiple of
    49 * 2^8 below 2^24 of them.  The result must be the BF16 rounding of the oracle's
    exact sum, bit for bit: every layout of codes and block scales has to be right."""
    rng = np.random.default_rng(21)
    M, N, K = 100, 384, 512

    def rows(R):
        codes = rng.integers(0, 16, size=(R, K)).astype(np.uint8)
        sfc = rng.choice(np.array([0x76, 0x7E], dtype=np.uint8), size=(R, K // 16))
        sfc[:, 5] = 0x7E                                    # 448: every row's maximum block
        for b in range(K // 16):
            codes[np.arange(R), 16 * b + rng.integers(0, 16, size=R)] = 7 | (rng.integers(0, 2, size=R) << 3)
        vals = np.where(codes & 8, -1.0, 1.0) * np.array([0, .5, 1, 1.5, 2, 3, 4, 6])[codes & 7]
        sv = torch.from_numpy(sfc).view(torch.float8_e4m3fn).double().numpy()
        e = rng.integers(-3, 3, size=(R, 1)).astype(np.float64)
        return vals * np.repeat(sv, 16, axis=1) * 2.0 ** e

    x, w = rows(M), rows(N)
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    wt = torch.from_numpy(w).to(torch.bfloat16).cuda()
    assert np.array_equal(xt.double().cpu().numpy(), x) and np.array_equal(wt.double().cpu().numpy(), w)
    qx, sfx, gx, qxr, sfxr, gxr = check_quant(fp8lib, oracle, xt)
    qw, sfw, gw, qwr, sfwr, gwr = check_quant(fp8lib, oracle, wt)
    exact = oracle.gemm_nvfp4(qxr, sfxr, gxr, qwr, sfwr, gwr)
    assert np.array_equal(exact, x @ w.T)                   # the construction round-trips
    want = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16)
    for splits in (1, 2):
        y = fp8lib.gemm_nvfp4(qx, sfx, gx, qw, sfw, gw, splits=splits).cpu().view(torch.int16)
        bad = (y != want).sum().item()
        assert bad == 0, f"splits={splits}: {bad} of {y.numel()} differ"


def test_linear_nvfp4_is_quantize_then_gemm(fp8lib, oracle):
    M, N, K = 64, 1536, 3584
    x = synth.normal_bf16((M, K), 1.0, 5, "cuda", outlier_channels=3, outlier_scale=30.0)
    w = synth.normal_bf16((N, K), 0.02, 6, "cuda")
    qw, sfw, gw = fp8lib.quantize_nvfp4(w)
    y, qx, sfx, gx = fp8lib.linear_nvfp4(x, qw, sfw, gw)
    qx2, sfx2, gx2 = fp8lib.quantize_nvfp4(x)
    assert torch.equal(qx, qx2) and torch.equal(sfx, sfx2) and torch.equal(gx.view(torch.int32), gx2.view(torch.int32))
    y2 = fp8lib.gemm_nvfp4(qx2, sfx2, gx2, qw, sfw, gw)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    qxr, sfxr, gxr = oracle.quantize_nvfp4(bits16(x))
    qwr, sfwr, gwr = oracle.quantize_nvfp4(bits16(w))
    gemm_tolerance_check(bits16(y), oracle.gemm_nvfp4(qxr, sfxr, gxr, qwr, sfwr, gwr), "linear_nvfp4")


# Qwen2.5-7B decode linears at full size: the weight quantization bit-exact, the outputs on
# 4096 sampled positions plus two full rows and two full columns
@pytest.mark.parametrize("M,N,K", [(64, 37888, 3584), (256, 3584, 18944), (128, 4608, 3584)])
def test_gemm_nvfp4_full_size_sampled(fp8lib, oracle, M, N, K):
    dev, ref, _ = operands(fp8lib, oracle, M, N, K, N + M)
    y = fp8lib.gemm_nvfp4(*dev)
    yb = bits16(y)
    rng = np.random.default_rng(M)
    m = np.concatenate([rng.integers(0, M, 4096), np.full(N, 3), np.full(N, M - 1),
                        np.arange(M), np.arange(M)])
    n = np.concatenate([rng.integers(0, N, 4096), np.arange(N), np.arange(N), np.full(M, 0), np.full(M, N - 1)])
    y_ref = oracle.gemm_nvfp4_sampled(*ref, m, n)
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    gemm_tolerance_check(yb[m, n], y_ref, f"nvfp4 {M}x{N}x{K}", rms=rms)


def test_nvfp4_linear_error_against_fp8(fp8lib, capsys):
    """The rollout formats' error on the same BF16 operands (activation with outlier
    channels, weights sigma 0.015): relative Frobenius error of the FP8 linear (1x128
    activations, 128x128 weight blocks) and of the NVFP4 linear, both against the exact
    product of the BF16 inputs.  NVFP4 keeps 1 mantissa bit against E4M3's 3, so its
    error is the larger, and both stay bounded."""
    M, N, K = 64, 2048, 3584
    x = synth.normal_bf16((M, K), 1.0, 31, "cuda", outlier_channels=4, outlier_scale=30.0)
    w = synth.normal_bf16((N, K), 0.015, 32, "cuda")
    exact = x.double().cpu() @ w.double().cpu().T
    qw8, sw8, _ = fp8lib.quantize_128x128(w)
    y8, _, _ = fp8lib.linear_fwd(x, qw8, sw8)
    q4, sf4, g4 = fp8lib.quantize_nvfp4(w)
    y4, _, _, _ = fp8lib.linear_nvfp4(x, q4, sf4, g4)
    err = lambda y: float(torch.linalg.norm(y.double().cpu() - exact) / torch.linalg.norm(exact))
    e8, e4 = err(y8), err(y4)
    with capsys.disabled():
        print(f"\nrelative Frobenius error vs the BF16 product: FP8 {e8:.3e}, NVFP4 {e4:.3e}")
    assert e8 < e4 < 0.2 and e8 < 0.05
