"""Pins of the oracle's block-scaled GEMM (forward, DGrad, WGrad index forms).

Scheme: "Technical summary: Jet-RL", section "Quantization Scheme" -- forward, DGrad and
WGrad GEMMs in FP8 on 1x128 / 128x128 / 128x1 quantized operands.  Independent checks:
  * exactly representable operands: quantization is the identity, so the oracle's
    block-scaled sum must equal numpy's float64 matmul of the original values bit for
    bit (the products and sums are exact in binary64 at these sizes);
  * torch CPU float64 matmul of the dequantized operands (a library routine) agrees to
    1e-12 relative for random data, in all three scale-index forms;
  * Y(2^a X, 2^b W) = 2^(a+b) Y exactly and Y(-X, W) = -Y.
A transposed operand, a swapped scale index or a dropped block fails one of these.
"""
import numpy as np
import pytest
import torch

POS_CODES = np.array([c for c in range(1, 0x7F)], dtype=np.uint8)


def bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_matrix(oracle, rng, shape, group_shape, jrange):
    """Values E4M3-grid * 2^j, one j per group, each group's max |value| = 448 * 2^j.
    Grid points drawn from the small codes keep all sums exact in binary64."""
    R, C = shape
    gr, gc = group_shape
    codes = rng.choice(POS_CODES[:40], size=shape) | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    x = oracle.e4m3_decode(codes)
    for r0 in range(0, R, gr):
        for c0 in range(0, C, gc):
            j = int(rng.integers(*jrange))
            blk = x[r0:r0 + gr, c0:c0 + gc]
            blk[rng.integers(0, blk.shape[0]), rng.integers(0, blk.shape[1])] = 448.0
            x[r0:r0 + gr, c0:c0 + gc] = blk * 2.0 ** j
    return x


def deq_rows(oracle, q, s):          # 1x128 along columns, s [C/128, R]
    return oracle.e4m3_decode(q) * np.repeat(s.T.astype(np.float64), 128, axis=1)


def deq_blocks(oracle, q, s):        # 128x128, s [N/128, K/128]
    S = np.kron(s.astype(np.float64), np.ones((128, 128)))
    return oracle.e4m3_decode(q) * S


def test_forward_exact_equals_float64_matmul(oracle):
    rng = np.random.default_rng(10)
    M, N, K = 96, 256, 384
    x = exact_matrix(oracle, rng, (M, K), (1, 128), (-4, 4))
    w = exact_matrix(oracle, rng, (N, K), (128, 128), (-4, 4))
    qx, sx = oracle.quantize_1x128(bf16_bits(x))
    qw, sw, _ = oracle.quantize_128x128(bf16_bits(w))
    assert np.array_equal(oracle.e4m3_decode(qx) * np.repeat(sx.T, 128, axis=1), x)
    y = oracle.gemm(qx, sx, qw, sw, "fwd")
    assert np.array_equal(y, x @ w.T)


def test_dgrad_exact_equals_float64_matmul(oracle):
    rng = np.random.default_rng(11)
    M, N, K = 64, 384, 256          # dY [M,N], W [N,K] -> dX [M,K], reduction over N
    dy = exact_matrix(oracle, rng, (M, N), (1, 128), (-4, 4))
    w = exact_matrix(oracle, rng, (N, K), (128, 128), (-4, 4))
    qdy, sdy = oracle.quantize_1x128(bf16_bits(dy))
    _, sw, qwT = oracle.quantize_128x128(bf16_bits(w))
    dx = oracle.gemm(qdy, sdy, qwT, sw, "dgrad")
    assert np.array_equal(dx, dy @ w)


def test_wgrad_exact_equals_float64_matmul(oracle):
    rng = np.random.default_rng(12)
    M, N, K = 256, 128, 384         # dY [M,N], X [M,K] -> dW [N,K], reduction over M
    dy = exact_matrix(oracle, rng, (M, N), (128, 1), (-4, 4))
    x = exact_matrix(oracle, rng, (M, K), (128, 1), (-4, 4))
    qdyT, sdyT = oracle.quantize_128x1(bf16_bits(dy))
    qxT, sxT = oracle.quantize_128x1(bf16_bits(x))
    dw = oracle.gemm(qdyT, sdyT, qxT, sxT, "wgrad")
    assert np.array_equal(dw, dy.T @ x)


@pytest.mark.parametrize("mode", ["fwd", "dgrad", "wgrad"])
def test_random_vs_torch_float64_dequantized(oracle, mode):
    rng = np.random.default_rng(20 + ["fwd", "dgrad", "wgrad"].index(mode))
    if mode == "fwd":
        M, N, K = 70, 256, 512
        x = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, (M, 1)))).astype(np.float32)
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        qa, sa = oracle.quantize_1x128(bf16_bits(x))
        qb, sb, _ = oracle.quantize_128x128(bf16_bits(w))
        A = deq_rows(oracle, qa, sa)
        B = deq_blocks(oracle, qb, sb)
        ref = torch.from_numpy(A) @ torch.from_numpy(B).T
        y = oracle.gemm(qa, sa, qb, sb, "fwd")
    elif mode == "dgrad":
        M, N, K = 64, 384, 256
        dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        qa, sa = oracle.quantize_1x128(bf16_bits(dy))
        qw, sb, qb = oracle.quantize_128x128(bf16_bits(w))
        A = deq_rows(oracle, qa, sa)
        W = deq_blocks(oracle, qw, sb)
        ref = torch.from_numpy(A) @ torch.from_numpy(W)
        y = oracle.gemm(qa, sa, qb, sb, "dgrad")
    else:
        M, N, K = 384, 128, 256
        dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
        x = rng.standard_normal((M, K)).astype(np.float32)
        qa, sa = oracle.quantize_128x1(bf16_bits(dy))
        qb, sb = oracle.quantize_128x1(bf16_bits(x))
        A = oracle.e4m3_decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)  # dY^T
        B = oracle.e4m3_decode(qb) * np.repeat(sb.T.astype(np.float64), 128, axis=1)  # X^T
        ref = torch.from_numpy(A) @ torch.from_numpy(B).T
        y = oracle.gemm(qa, sa, qb, sb, "wgrad")
    ref = ref.numpy()
    scale = np.abs(ref).max()
    assert np.max(np.abs(y - ref)) <= 1e-12 * scale


def test_scaling_law_and_sign(oracle):
    rng = np.random.default_rng(30)
    M, N, K = 32, 128, 256
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xb, wb = bf16_bits(x), bf16_bits(w)
    qx, sx = oracle.quantize_1x128(xb)
    qw, sw, _ = oracle.quantize_128x128(wb)
    y0 = oracle.gemm(qx, sx, qw, sw, "fwd")
    xf, wf = oracle.bf16_to_f32(xb), oracle.bf16_to_f32(wb)
    for a, b in ((3, -2), (-7, 5)):
        qx2, sx2 = oracle.quantize_1x128(bf16_bits(xf * np.float32(2.0 ** a)))
        qw2, sw2, _ = oracle.quantize_128x128(bf16_bits(wf * np.float32(2.0 ** b)))
        y = oracle.gemm(qx2, sx2, qw2, sw2, "fwd")
        assert np.array_equal(y, y0 * 2.0 ** (a + b))
    qxn, sxn = oracle.quantize_1x128(bf16_bits(-xf))
    assert np.array_equal(oracle.gemm(qxn, sxn, qw, sw, "fwd"), -y0)


def test_sampled_matches_full(oracle):
    rng = np.random.default_rng(31)
    M, N, K = 50, 256, 384
    qx, sx = oracle.quantize_1x128(bf16_bits(rng.standard_normal((M, K))))
    qw, sw, _ = oracle.quantize_128x128(bf16_bits(rng.standard_normal((N, K)) * 0.02))
    y = oracle.gemm(qx, sx, qw, sw, "fwd")
    r1 = rng.integers(0, M, 300)
    r2 = rng.integers(0, N, 300)
    assert np.array_equal(oracle.gemm_sampled(qx, sx, qw, sw, "fwd", r1, r2), y[r1, r2])
