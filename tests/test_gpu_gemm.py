"""Block-scaled FP8 GEMMs on the GPU vs the CPU oracle.

"Technical summary: Jet-RL", section "Quantization Scheme": forward, DGrad and WGrad run
in FP8 (1x128 activations/gradients, 128x128 weights, 128x1 WGrad operands); section "Core
architecture": the rollout (decode-shaped, split-K) kernel shares the training forward
pass's numerics.  Every output element must satisfy
    |y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref)
against the oracle's unrounded binary64 result on the same codes and scales.  The codes
come from the oracle-checked GPU quantizers and are re-derived on the host by the oracle,
so both sides see identical operands.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth
from parity import assert_same_bits_f32, assert_same_u8, bits16, f32, gemm_tolerance_check, u8

pytestmark = pytest.mark.gpu


def fwd_operands(fp8lib, oracle, M, N, K, seed):
    x = synth.normal_bf16((M, K), 1.0, seed, "cuda", outlier_channels=max(1, K // 1000),
                          outlier_scale=30.0)
    w = synth.normal_bf16((N, K), 0.02, seed + 1, "cuda")
    qx, sx = fp8lib.quantize_1x128(x)
    qw, sw, qwT = fp8lib.quantize_128x128(w)
    # the host sees the same operands: re-derive them with the oracle and compare
    qxr, sxr = oracle.quantize_1x128(bits16(x))
    assert_same_u8(u8(qx), qxr, "qx")
    assert_same_bits_f32(f32(sx), sxr, "sx")
    return qx, sx, qw, sw, qwT


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512), (300, 384, 640),
                                   (1000, 1280, 1024), (129, 128, 256)])
def test_fwd_tiled(fp8lib, oracle, M, N, K):
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, M + N + K)
    y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_TILED)
    y_ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    gemm_tolerance_check(bits16(y), y_ref, f"fwd {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 5, 64, 100, 128, 200, 256])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fwd_decode(fp8lib, oracle, M, splits):
    N, K = 1280, 1024
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 7 * M + splits)
    y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_SPLITK, splits=splits)
    y_ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    gemm_tolerance_check(bits16(y), y_ref, f"decode M={M} splits={splits}")
    # deterministic: the same call gives the same bytes
    y2 = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_SPLITK, splits=splits)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


# decode form with the weights on the MMA's M side: token counts around every padding class
# (32/64/128/256), cluster sizes from one CTA to one K-block per CTA
@pytest.mark.parametrize("M", [1, 5, 31, 32, 33, 64, 100, 128, 129, 200, 256])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_fwd_decode_swapped(fp8lib, oracle, M, splits):
    N, K = 1280, 1024
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 11 * M + splits)
    y_ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_DECODE, splits=splits)
    gemm_tolerance_check(bits16(y), y_ref, f"decode (swapped) M={M} splits={splits}")
    y2 = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_DECODE, splits=splits)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert fp8lib.check_status() == _abi.FP8RL_OK


@pytest.mark.parametrize("M,N,K", [(64, 1280, 3584), (256, 768, 2048), (17, 2048, 512), (300, 512, 1024),
                                   (1, 1280, 1024), (31, 768, 512), (33, 1280, 2048), (100, 4608, 1024),
                                   (128, 3584, 3584), (64, 37888, 3584), (256, 37888, 3584)])
def test_linear_fwd_quantizes_and_multiplies(fp8lib, oracle, M, N, K):
    """The fused linear: its activation codes and scales are the oracle's 1x128 quantization
    bit for bit, and its output is within the GEMM bound of the oracle's result from them
    and byte-identical to the GEMM the automatic choice runs on those codes."""
    x = synth.normal_bf16((M, K), 1.0, M + K + 5, "cuda", outlier_channels=3, outlier_scale=30.0)
    w = synth.normal_bf16((N, K), 0.02, N + 7, "cuda")
    qw, sw, _ = fp8lib.quantize_128x128(w, transpose=False)
    for rep in range(2):
        y, qx, sx = fp8lib.linear_fwd(x, qw, sw)
        qxr, sxr = oracle.quantize_1x128(bits16(x))
        assert_same_u8(u8(qx), qxr, "qx")
        assert_same_bits_f32(f32(sx), sxr, "sx")
        if M * N * K <= 1 << 31:
            y_ref = oracle.gemm(qxr, sxr, u8(qw), f32(sw), "fwd")
            gemm_tolerance_check(bits16(y), y_ref, f"linear {M}x{N}x{K} rep {rep}")
        # the GEMM the automatic choice runs on the same codes gives the same bytes
        y2 = fp8lib.gemm_fwd(qx, sx, qw, sw)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), f"linear {M}x{N}x{K}"
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_linear_fwd_strided_activation(fp8lib, oracle):
    """The fused linear reads x with its row stride (a column slice of a wider buffer), at a
    token count inside the 64-token padding class of the decode form."""
    M, N, K = 40, 2048, 1536
    big = synth.normal_bf16((M, K + 384), 1.0, 123, "cuda", outlier_channels=4, outlier_scale=30.0)
    x = big[:, 128:128 + K]
    w = synth.normal_bf16((N, K), 0.02, 124, "cuda")
    qw, sw, _ = fp8lib.quantize_128x128(w, transpose=False)
    y, qx, sx = fp8lib.linear_fwd(x, qw, sw)
    qxr, sxr = oracle.quantize_1x128(bits16(x.contiguous()))
    assert_same_u8(u8(qx), qxr, "qx")
    assert_same_bits_f32(f32(sx), sxr, "sx")
    y_ref = oracle.gemm(qxr, sxr, u8(qw), f32(sw), "fwd")
    gemm_tolerance_check(bits16(y), y_ref, "strided linear")
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_fwd_auto_matches_forms(fp8lib, oracle):
    """AUTO picks the decode form for M <= 256; both forms obey the same bound."""
    M, N, K = 192, 768, 2048
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 99)
    y_ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    for v in (_abi.FP8RL_VARIANT_AUTO, _abi.FP8RL_VARIANT_TILED, _abi.FP8RL_VARIANT_SPLITK,
              _abi.FP8RL_VARIANT_PAIR, _abi.FP8RL_VARIANT_DECODE, _abi.FP8RL_VARIANT_MULTICAST):
        gemm_tolerance_check(bits16(fp8lib.gemm_fwd(qx, sx, qw, sw, variant=v)), y_ref, f"variant {v}")


# (256, 640, 512) and (200, 768, 1024): 5 and 6 K-blocks of reduction with B's block scales
# stored [K-block][column block] in rows of 4 and 8 blocks, so the copy warp fetches them by
# TMA in groups of 4 K-blocks and the last group of each tile is partial.
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (300, 384, 512), (512, 1024, 768),
                                   (256, 640, 512), (200, 768, 1024)])
def test_dgrad(fp8lib, oracle, M, N, K):
    dy = synth.normal_bf16((M, N), 1e-3, M + 3, "cuda")
    w = synth.normal_bf16((N, K), 0.02, K + 5, "cuda")
    qdy, sdy = fp8lib.quantize_1x128(dy)
    _, sw, qwT = fp8lib.quantize_128x128(w)
    dx = fp8lib.gemm_dgrad(qdy, sdy, qwT, sw)
    ref = oracle.gemm(u8(qdy), f32(sdy), u8(qwT), f32(sw), "dgrad")
    gemm_tolerance_check(bits16(dx), ref, f"dgrad {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (1024, 256, 768)])
def test_wgrad(fp8lib, oracle, M, N, K):
    dy = synth.normal_bf16((M, N), 1e-3, M + 11, "cuda")
    x = synth.normal_bf16((M, K), 1.0, K + 13, "cuda", outlier_channels=2, outlier_scale=30.0)
    qdyT, sdyT = fp8lib.quantize_128x1(dy)
    qxT, sxT = fp8lib.quantize_128x1(x)
    dw = fp8lib.gemm_wgrad(qdyT, sdyT, qxT, sxT)
    ref = oracle.gemm(u8(qdyT), f32(sdyT), u8(qxT), f32(sxT), "wgrad")
    gemm_tolerance_check(bits16(dw), ref, f"wgrad {M}x{N}x{K}")


def test_exactly_representable_gemm(fp8lib, oracle):
    """Operands on the E4M3 grid with power-of-two scales: quantization is the identity and
    the exact product is numpy's float64 matmul; the GPU must be within BF16 rounding."""
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 512
    codes_x = rng.integers(0x20, 0x48, size=(M, K)).astype(np.uint8) | (rng.integers(0, 2, (M, K)).astype(np.uint8) << 7)
    codes_w = rng.integers(0x20, 0x48, size=(N, K)).astype(np.uint8) | (rng.integers(0, 2, (N, K)).astype(np.uint8) << 7)
    x = oracle.e4m3_decode(codes_x)
    w = oracle.e4m3_decode(codes_w)
    x[:, ::128] = 448.0          # every 1x128 group has max 448 -> scale 1
    w[::128, ::128] = 448.0      # every 128x128 block has max 448 -> scale 1
    xt = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).cuda()
    wt = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).cuda()
    qx, sx = fp8lib.quantize_1x128(xt)
    qw, sw, _ = fp8lib.quantize_128x128(wt)
    assert torch.all(sx == 1.0) and torch.all(sw == 1.0)
    exact = x @ w.T
    for v in (_abi.FP8RL_VARIANT_TILED, _abi.FP8RL_VARIANT_SPLITK, _abi.FP8RL_VARIANT_PAIR,
              _abi.FP8RL_VARIANT_DECODE, _abi.FP8RL_VARIANT_MULTICAST):
        y = bits16(fp8lib.gemm_fwd(qx, sx, qw, sw, variant=v))
        yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.all(np.abs(yf - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-30)


def test_scaling_law_on_device(fp8lib, oracle):
    """Y(2^a X, 2^b W) = 2^(a+b) Y: the scales absorb powers of two exactly."""
    M, N, K = 256, 512, 1024
    x = synth.normal_bf16((M, K), 1.0, 21, "cuda")
    w = synth.normal_bf16((N, K), 0.02, 22, "cuda")
    qx, sx = fp8lib.quantize_1x128(x)
    qw, sw, _ = fp8lib.quantize_128x128(w)
    qx2, sx2 = fp8lib.quantize_1x128((x.float() * 8.0).to(torch.bfloat16))
    qw2, sw2, _ = fp8lib.quantize_128x128((w.float() * 0.25).to(torch.bfloat16))
    for v in (_abi.FP8RL_VARIANT_TILED, _abi.FP8RL_VARIANT_SPLITK, _abi.FP8RL_VARIANT_PAIR,
              _abi.FP8RL_VARIANT_DECODE, _abi.FP8RL_VARIANT_MULTICAST):
        y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=v).float()
        y2 = fp8lib.gemm_fwd(qx2, sx2, qw2, sw2, variant=v).float()
        assert torch.equal(y2, y * 2.0)


@pytest.mark.parametrize("variant", [_abi.FP8RL_VARIANT_TILED, _abi.FP8RL_VARIANT_PAIR,
                                     _abi.FP8RL_VARIANT_MULTICAST])
def test_tiled_deterministic_and_grid_independent(fp8lib, oracle, variant):
    """Both persistent forms against the oracle, with a full grid and with a few CTAs (or
    clusters) that each walk many tiles; the two runs give the same bytes."""
    M, N, K = 640, 1536, 1024
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 3)
    ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    y1 = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=variant)
    y2 = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=variant, grid=7)
    gemm_tolerance_check(bits16(y1), ref, f"variant {variant}, full grid")
    gemm_tolerance_check(bits16(y2), ref, f"variant {variant}, grid 7")
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


# ------------------------------------------------------------------ paired-SM form
# 256 x 128 and 256 x 256 output tiles on clusters of two CTAs.  Row counts that are not
# multiples of 256 leave the second CTA of the last pair partly or wholly outside A, and
# column counts that are not multiples of the tile width leave B's second half partly or
# wholly outside B (TMA zero fill, clipped stores); grid = clusters, so small grids make
# each cluster walk many tiles.

@pytest.mark.parametrize("M,N,K", [(256, 128, 512), (128, 256, 512), (300, 384, 512),
                                   (1000, 1280, 1024), (132, 128, 2048), (520, 640, 1536)])
@pytest.mark.parametrize("epi", [8, 16])
@pytest.mark.parametrize("pn", [128, 256])
def test_fwd_pair(fp8lib, oracle, M, N, K, epi, pn):
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, M + N + K + epi)
    ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    for grid in (0, 2):
        y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_PAIR, epi_warps=epi, grid=grid, tile_n=pn)
        gemm_tolerance_check(bits16(y), ref, f"pair fwd {M}x{N}x{K} epi {epi} grid {grid} tile {pn}")
    assert fp8lib.check_status() == _abi.FP8RL_OK


# (512, 640, 512): 5 K-blocks, the last scale group of each tile partial
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (300, 384, 1024), (512, 640, 512),
                                   (768, 1024, 2048)])
def test_dgrad_pair(fp8lib, oracle, M, N, K):
    dy = synth.normal_bf16((M, N), 1e-3, M + 31, "cuda")
    w = synth.normal_bf16((N, K), 0.02, K + 35, "cuda")
    qdy, sdy = fp8lib.quantize_1x128(dy)
    _, sw, qwT = fp8lib.quantize_128x128(w)
    ref = oracle.gemm(u8(qdy), f32(sdy), u8(qwT), f32(sw), "dgrad")
    for v, grid, pn in ((_abi.FP8RL_VARIANT_PAIR, 0, 128), (_abi.FP8RL_VARIANT_PAIR, 3, 128),
                        (_abi.FP8RL_VARIANT_PAIR, 0, 256), (_abi.FP8RL_VARIANT_PAIR, 3, 256),
                        (_abi.FP8RL_VARIANT_TILED, 0, 0)):
        dx = fp8lib.gemm_dgrad(qdy, sdy, qwT, sw, variant=v, grid=grid, tile_n=pn)
        gemm_tolerance_check(bits16(dx), ref, f"dgrad {M}x{N}x{K} variant {v} grid {grid} tile {pn}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (1024, 256, 768),
                                   (384, 640, 1152)])
@pytest.mark.parametrize("epi", [8, 16])
@pytest.mark.parametrize("pn", [128, 256])
def test_wgrad_pair(fp8lib, oracle, M, N, K, epi, pn):
    dy = synth.normal_bf16((M, N), 1e-3, M + 41 + epi, "cuda")
    x = synth.normal_bf16((M, K), 1.0, K + 43, "cuda", outlier_channels=2, outlier_scale=30.0)
    qdyT, sdyT = fp8lib.quantize_128x1(dy)
    qxT, sxT = fp8lib.quantize_128x1(x)
    ref = oracle.gemm(u8(qdyT), f32(sdyT), u8(qxT), f32(sxT), "wgrad")
    for grid in (0, 2):
        dw = fp8lib.gemm_wgrad(qdyT, sdyT, qxT, sxT, variant=_abi.FP8RL_VARIANT_PAIR, epi_warps=epi, grid=grid,
                               tile_n=pn)
        gemm_tolerance_check(bits16(dw), ref, f"pair wgrad {M}x{N}x{K} epi {epi} grid {grid} tile {pn}")
    dw = fp8lib.gemm_wgrad(qdyT, sdyT, qxT, sxT, variant=_abi.FP8RL_VARIANT_TILED)
    gemm_tolerance_check(bits16(dw), ref, f"one-SM wgrad {M}x{N}x{K}")


# ------------------------------------------------------------------ multicast form
# Clusters of two CTAs on vertically adjacent 128 x 256 tiles share each B tile (each CTA
# copies half of it into both).  Odd m-tile counts leave the second CTA of the last pair
# wholly outside A (zero fill, clipped stores); N not a multiple of 256 leaves the second
# half of the last B tile outside B; grid = clusters.

@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (384, 384, 512), (300, 1280, 1024),
                                   (132, 128, 2048), (1000, 768, 1536)])
def test_fwd_multicast(fp8lib, oracle, M, N, K):
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 3 * M + N + K)
    ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    for grid in (0, 1, 3):
        y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_MULTICAST, grid=grid)
        gemm_tolerance_check(bits16(y), ref, f"multicast fwd {M}x{N}x{K} grid {grid}")
    assert fp8lib.check_status() == _abi.FP8RL_OK


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (300, 384, 1024), (512, 640, 512)])
def test_dgrad_multicast(fp8lib, oracle, M, N, K):
    dy = synth.normal_bf16((M, N), 1e-3, M + 61, "cuda")
    w = synth.normal_bf16((N, K), 0.02, K + 65, "cuda")
    qdy, sdy = fp8lib.quantize_1x128(dy)
    _, sw, qwT = fp8lib.quantize_128x128(w)
    ref = oracle.gemm(u8(qdy), f32(sdy), u8(qwT), f32(sw), "dgrad")
    for grid in (0, 2):
        dx = fp8lib.gemm_dgrad(qdy, sdy, qwT, sw, variant=_abi.FP8RL_VARIANT_MULTICAST, grid=grid)
        gemm_tolerance_check(bits16(dx), ref, f"multicast dgrad {M}x{N}x{K} grid {grid}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (1024, 384, 768),
                                   (384, 640, 1152)])
def test_wgrad_multicast(fp8lib, oracle, M, N, K):
    dy = synth.normal_bf16((M, N), 1e-3, M + 71, "cuda")
    x = synth.normal_bf16((M, K), 1.0, K + 73, "cuda", outlier_channels=2, outlier_scale=30.0)
    qdyT, sdyT = fp8lib.quantize_128x1(dy)
    qxT, sxT = fp8lib.quantize_128x1(x)
    ref = oracle.gemm(u8(qdyT), f32(sdyT), u8(qxT), f32(sxT), "wgrad")
    for grid in (0, 2):
        dw = fp8lib.gemm_wgrad(qdyT, sdyT, qxT, sxT, variant=_abi.FP8RL_VARIANT_MULTICAST, grid=grid)
        gemm_tolerance_check(bits16(dw), ref, f"multicast wgrad {M}x{N}x{K} grid {grid}")
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_multicast_same_bytes_as_one_sm_form(fp8lib, oracle):
    """The multicast form changes only where B's bytes come from: the same partial sums in
    the same order, so the same BF16 output bytes as the one-SM form."""
    M, N, K = 640, 1536, 1024
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 17)
    y1 = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_TILED)
    y2 = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_MULTICAST)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_pair_refuses_scales_it_cannot_copy(fp8lib, oracle):
    """PAIR needs TMA-able scale rows; AUTO then takes the one-SM form."""
    M, N, K = 256, 256, 640      # 5 K-blocks: rows of 5 block scales are not 16-byte multiples
    qx, sx, qw, sw, _ = fwd_operands(fp8lib, oracle, M, N, K, 77)
    with pytest.raises(_abi.Fp8rlError) as e:
        fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_PAIR)
    assert e.value.status == _abi.FP8RL_ERR_SHAPE
    ref = oracle.gemm(u8(qx), f32(sx), u8(qw), f32(sw), "fwd")
    gemm_tolerance_check(bits16(fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_AUTO)), ref, "auto")
