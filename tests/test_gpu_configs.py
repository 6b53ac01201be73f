"""Parity at the full sizes of the five workloads, through the same entry points and kernel
choices the benchmark times (automatic variants).

Quantizers are compared bit for bit against the CPU oracle: whole tensors where the oracle
finishes in seconds, otherwise every group of a seeded sample of rows (1x128 groups) and of
column blocks (128x1 groups).  GEMMs are compared on 4096 seeded random output elements
plus two full rows and two full columns, against the oracle's unrounded binary64 value
computed one element at a time, with the elementwise bound
|y - y_ref| <= 2^-7 |y_ref| + 1e-3 rms(y_ref) (rms over the sampled set).

Workloads ("Technical summary: Jet-RL", section "Experimental results", evaluates
Llama3.1-8B, Qwen2.5-7B and Qwen3-8B-Base RL runs; their linear-layer shapes, 8k-16k
tokens, stand in for the datasets, which are not used): see block_scaled_fp8_x1_gb300/synth.py.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth
from parity import (assert_same_bits_f32, assert_same_u8, bits16, f32, gemm_tolerance_check,
                    silu_group_matches, u8)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def sample_positions(R1, R2, seed, n=4096):
    rng = np.random.default_rng(seed)
    r1 = [rng.integers(0, R1, n)]
    r2 = [rng.integers(0, R2, n)]
    for row in rng.integers(0, R1, 2):
        r1.append(np.full(R2, row))
        r2.append(np.arange(R2))
    for col in rng.integers(0, R2, 2):
        r1.append(np.arange(R1))
        r2.append(np.full(R1, col))
    return np.concatenate(r1).astype(np.int64), np.concatenate(r2).astype(np.int64)


def check_gemm_sampled(oracle, y, A, sa, B, sb, mode, seed, what):
    R1, R2 = y.shape
    r1, r2 = sample_positions(R1, R2, seed)
    ref = oracle.gemm_sampled(A, sa, B, sb, mode, r1, r2)
    i1 = torch.from_numpy(r1).to(y.device)
    i2 = torch.from_numpy(r2).to(y.device)
    yb = bits16(y[i1, i2])
    return gemm_tolerance_check(yb, ref, what)


def check_1x128_rows(oracle, x, q, s, rows, what):
    """Every 1x128 group of the given rows of x [M, K]."""
    idx = torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(x.device)
    xr = bits16(x[idx])
    qr, sr = oracle.quantize_1x128(xr)
    assert_same_u8(u8(q[idx]), qr, what + " codes")
    assert_same_bits_f32(f32(s[:, idx]), sr, what + " scales")


def check_128x1_blocks(oracle, x, qT, sT, blocks, cols, what):
    """The 128x1 groups of the given (row block, column) pairs of x [M, K]."""
    xb = bits16(x)
    qTh, sTh = u8(qT), f32(sT)
    for b, k in zip(blocks, cols):
        vals = oracle.bf16_to_f32(xb[b * 128:(b + 1) * 128, k])
        qg, sg = oracle.quant_group(vals)
        assert np.array_equal(qTh[k, b * 128:(b + 1) * 128], qg), (what, b, k)
        assert np.float32(sTh[b, k]).view(np.uint32) == np.float32(sg).view(np.uint32), (what, b, k)


# ------------------------------------------------------------------ single linear

def test_single_linear_256x512(fp8lib, oracle):
    w = synth.SINGLE_LINEAR_256x512
    lin = w.linears[0]
    x = synth.activation(w, 256, lin.K, 0, DEV)
    wt = synth.weight(w, lin, 1, DEV)
    qx, sx = fp8lib.quantize_1x128(x)
    qw, sw, _ = fp8lib.quantize_128x128(wt)
    qxr, sxr = oracle.quantize_1x128(bits16(x))
    qwr, swr, _ = oracle.quantize_128x128(bits16(wt))
    assert_same_u8(u8(qx), qxr, "X codes")
    assert_same_bits_f32(f32(sx), sxr, "X scales")
    assert_same_u8(u8(qw), qwr, "W codes")
    assert_same_bits_f32(f32(sw), swr, "W scales")
    ref = oracle.gemm(qxr, sxr, qwr, swr, "fwd")
    for v in (_abi.FP8RL_VARIANT_AUTO, _abi.FP8RL_VARIANT_TILED):
        y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=v)
        gemm_tolerance_check(bits16(y), ref, f"single linear variant {v}")


# ------------------------------------------------------------------ Llama-3.1-8B MLP, 8192 tokens

@pytest.fixture(scope="module")
def llama_forward(fp8lib):
    w = synth.LLAMA8B_MLP_M8192
    gate_up, down = w.linears
    M = w.M[0]
    x = synth.activation(w, M, gate_up.K, 0, DEV)
    gamma = torch.ones(gate_up.K, dtype=torch.bfloat16, device=DEV)
    w_gu = synth.weight(w, gate_up, 1, DEV)
    w_d = synth.weight(w, down, 2, DEV)
    q_gu, s_gu, qT_gu = fp8lib.quantize_128x128(w_gu)
    q_d, s_d, qT_d = fp8lib.quantize_128x128(w_d)
    qx, sx, qxT, sxT, rstd = fp8lib.rmsnorm_quant(x, gamma, w.extra["eps"])
    gu = fp8lib.gemm_fwd(qx, sx, q_gu, s_gu)
    qh, sh, qhT, shT = fp8lib.silu_mul_quant(gu)
    y = fp8lib.gemm_fwd(qh, sh, q_d, s_d)
    torch.cuda.synchronize()
    return dict(w=w, x=x, gamma=gamma, w_gu=w_gu, w_d=w_d, q_gu=q_gu, s_gu=s_gu, qT_gu=qT_gu,
                q_d=q_d, s_d=s_d, qT_d=qT_d, qx=qx, sx=sx, qxT=qxT, sxT=sxT, rstd=rstd, gu=gu,
                qh=qh, sh=sh, qhT=qhT, shT=shT, y=y)


def test_llama_weight_quantization(fp8lib, oracle, llama_forward):
    f = llama_forward
    for name in ("gu", "d"):
        q, s, qT = f["q_" + name], f["s_" + name], f["qT_" + name]
        qr, sr, qTr = oracle.quantize_128x128(bits16(f["w_" + name]))
        assert_same_u8(u8(q), qr, f"W_{name} codes")
        assert_same_bits_f32(f32(s), sr, f"W_{name} scales")
        assert_same_u8(u8(qT), qTr, f"W_{name}^T codes")


def test_llama_rmsnorm_quant(fp8lib, oracle, llama_forward):
    f = llama_forward
    xb, gb = bits16(f["x"]), bits16(f["gamma"])
    _, _, _, _, r_ref, _ = oracle.rmsnorm_quant(xb, gb, f["w"].extra["eps"])
    r_gpu = f32(f["rstd"])
    diff = r_gpu.view(np.int32).astype(np.int64) - r_ref.view(np.int32).astype(np.int64)
    assert np.all(np.abs(diff) <= 1)
    qr, sr, qTr, sTr, _, _ = oracle.rmsnorm_quant(xb, gb, f["w"].extra["eps"], rstd_in=r_gpu)
    assert_same_u8(u8(f["qx"]), qr, "q")
    assert_same_bits_f32(f32(f["sx"]), sr, "s")
    assert_same_u8(u8(f["qxT"]), qTr, "qT")
    assert_same_bits_f32(f32(f["sxT"]), sTr, "sT")


def test_llama_gate_up_forward(fp8lib, oracle, llama_forward):
    f = llama_forward
    check_gemm_sampled(oracle, f["gu"], u8(f["qx"]), f32(f["sx"]), u8(f["q_gu"]), f32(f["s_gu"]),
                       "fwd", 1, "gate_up forward 8192x28672x4096")


def test_llama_silu_mul_quant_sampled(fp8lib, oracle, llama_forward):
    f = llama_forward
    gu = f["gu"]
    M, I2 = gu.shape
    I = I2 // 2
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(M, 512, replace=False))
    gub = bits16(gu[torch.from_numpy(rows).to(DEV)])
    h, alt, _ = oracle.silu_mul(gub)
    qr, sr = oracle.quantize_1x128(h)
    qg, sg = u8(f["qh"])[rows], f32(f["sh"])[:, rows]
    for i in range(len(rows)):
        for b in range(I // 128):
            sl = slice(b * 128, (b + 1) * 128)
            if np.array_equal(qg[i, sl], qr[i, sl]) and sg[b, i].view(np.uint32) == sr[b, i].view(np.uint32):
                continue
            assert silu_group_matches(oracle, qg[i, sl], sg[b, i], h[i, sl], alt[i, sl]), (rows[i], b)
    # 128x1 groups: a sample of whole row blocks
    blocks = rng.choice(M // 128, 4, replace=False)
    qTg, sTg = u8(f["qhT"]), f32(f["shT"])
    for blk in blocks:
        hb_gu = bits16(gu[blk * 128:(blk + 1) * 128])
        hb, altb, _ = oracle.silu_mul(hb_gu)
        qTr, sTr = oracle.quantize_128x1(hb)
        for i in range(I):
            sl = slice(blk * 128, (blk + 1) * 128)
            if np.array_equal(qTg[i, sl], qTr[i]) and sTg[blk, i].view(np.uint32) == sTr[0, i].view(np.uint32):
                continue
            assert silu_group_matches(oracle, qTg[i, sl], sTg[blk, i], hb[:, i], altb[:, i]), (blk, i)


def test_llama_down_forward(fp8lib, oracle, llama_forward):
    f = llama_forward
    check_gemm_sampled(oracle, f["y"], u8(f["qh"]), f32(f["sh"]), u8(f["q_d"]), f32(f["s_d"]),
                       "fwd", 2, "down forward 8192x4096x14336")


# ------------------------------------------------------------------ Llama MLP backward

def test_llama_backward(fp8lib, oracle, llama_forward):
    f = llama_forward
    wb = synth.LLAMA8B_MLP_BWD_M8192
    gate_up, down = wb.linears
    M = wb.M[0]
    for idx, (lin, qwT, sw, saved_qT, saved_sT) in enumerate(
            ((down, f["qT_d"], f["s_d"], f["qhT"], f["shT"]),
             (gate_up, f["qT_gu"], f["s_gu"], f["qxT"], f["sxT"]))):
        dy = synth.gradient(wb, M, lin.N, 3 + idx, DEV)
        qdy, sdy, qdyT, sdyT = fp8lib.quantize_1x128(dy, dual=True)
        rng = np.random.default_rng(10 + idx)
        check_1x128_rows(oracle, dy, qdy, sdy, np.sort(rng.choice(M, 256, replace=False)), f"dY_{lin.name}")
        check_128x1_blocks(oracle, dy, qdyT, sdyT, rng.integers(0, M // 128, 512),
                           rng.integers(0, lin.N, 512), f"dY_{lin.name} 128x1")
        dx = fp8lib.gemm_dgrad(qdy, sdy, qwT, sw)
        check_gemm_sampled(oracle, dx, u8(qdy), f32(sdy), u8(qwT), f32(sw), "dgrad", 20 + idx,
                           f"DGrad {lin.name}")
        dw = fp8lib.gemm_wgrad(qdyT, sdyT, saved_qT, saved_sT)
        check_gemm_sampled(oracle, dw, u8(qdyT), f32(sdyT), u8(saved_qT), f32(saved_sT), "wgrad",
                           30 + idx, f"WGrad {lin.name}")


# ------------------------------------------------------------------ Qwen2.5-7B decode

@pytest.mark.parametrize("M", [64, 128, 256])
def test_qwen7b_decode(fp8lib, oracle, M):
    w = synth.QWEN7B_DECODE
    for idx, lin in enumerate(w.linears):
        x = synth.activation(w, M, lin.K, 10 * idx, DEV)
        wt = synth.weight(w, lin, 10 * idx + 1, DEV)
        qx, sx = fp8lib.quantize_1x128(x)
        qw, sw, _ = fp8lib.quantize_128x128(wt, transpose=False)
        qxr, sxr = oracle.quantize_1x128(bits16(x))
        assert_same_u8(u8(qx), qxr, f"{lin.name} X codes")
        assert_same_bits_f32(f32(sx), sxr, f"{lin.name} X scales")
        y = fp8lib.gemm_fwd(qx, sx, qw, sw)       # automatic choice (gate_up at 256 tokens: the paired form)
        check_gemm_sampled(oracle, y, qxr, sxr, u8(qw), f32(sw), "fwd", 40 + idx,
                           f"decode {lin.name} M={M}")


# ------------------------------------------------------------------ Qwen2.5-32B layer, 16384 tokens

@pytest.mark.parametrize("which", ["qkv", "o", "gate_up", "down"])
def test_qwen32b_layer(fp8lib, oracle, which):
    w = synth.QWEN32B_LAYER_M16384
    idx = [l.name for l in w.linears].index(which)
    lin = w.linears[idx]
    M = w.M[0]
    rng = np.random.default_rng(50 + idx)
    x = synth.activation(w, M, lin.K, 10 * idx, DEV)
    wt = synth.weight(w, lin, 10 * idx + 1, DEV)
    dy = synth.gradient(w, M, lin.N, 10 * idx + 2, DEV)
    q, s, qT = fp8lib.quantize_128x128(wt)
    rows_w = np.sort(rng.choice(lin.N // 128, 2, replace=False))
    for bn in rows_w:
        qr, sr, _ = oracle.quantize_128x128(bits16(wt[bn * 128:(bn + 1) * 128]), with_transpose=False)
        assert_same_u8(u8(q[bn * 128:(bn + 1) * 128]), qr, f"W_{which} block row {bn}")
        assert_same_bits_f32(f32(s[bn:bn + 1]), sr, f"W_{which} scales {bn}")
    qx, sx, qxT, sxT = fp8lib.quantize_1x128(x, dual=True)
    check_1x128_rows(oracle, x, qx, sx, np.sort(rng.choice(M, 128, replace=False)), f"X_{which}")
    check_128x1_blocks(oracle, x, qxT, sxT, rng.integers(0, M // 128, 256),
                       rng.integers(0, lin.K, 256), f"X_{which} 128x1")
    y = fp8lib.gemm_fwd(qx, sx, q, s)
    check_gemm_sampled(oracle, y, u8(qx), f32(sx), u8(q), f32(s), "fwd", 60 + idx, f"fwd {which}")
    del y
    qdy, sdy, qdyT, sdyT = fp8lib.quantize_1x128(dy, dual=True)
    check_1x128_rows(oracle, dy, qdy, sdy, np.sort(rng.choice(M, 128, replace=False)), f"dY_{which}")
    dx = fp8lib.gemm_dgrad(qdy, sdy, qT, s)
    check_gemm_sampled(oracle, dx, u8(qdy), f32(sdy), u8(qT), f32(s), "dgrad", 70 + idx, f"dgrad {which}")
    del dx
    dw = fp8lib.gemm_wgrad(qdyT, sdyT, qxT, sxT)
    check_gemm_sampled(oracle, dw, u8(qdyT), f32(sdyT), u8(qxT), f32(sxT), "wgrad", 80 + idx,
                       f"wgrad {which}")
    assert fp8lib.check_status() == _abi.FP8RL_OK
