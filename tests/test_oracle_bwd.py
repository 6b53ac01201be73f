"""Pins of the oracle's backward steps next to the quantizers (test infrastructure).

"Technical summary: Jet-RL", section "Quantization Scheme": gradients between operators
stay BF16, DGrad / WGrad run in FP8 on quantized gradients; the operators either side of
the gradient quantizer are the SiLU-mul backward (producing the gradient of the gate_up
output) and the RMSNorm backward (from the forward's saved rstd).  Both are the chain rule
of the forward readings (SiLU-mul: h = silu(g) * u; RMSNorm: y = (x * rstd) * gamma), so
they are pinned here against references the oracle does not share:

  * central finite differences of the forward, evaluated independently in numpy binary64
    (scipy's logistic for the sigmoid),
  * closed forms at g = 0 and for constant RMSNorm rows,
  * dgamma as a numpy reduction.
A plausible mistake -- a dropped (1 + g(1 - s)) factor, a missing r^3 term, the gate / up
halves swapped, the wrong sign -- fails one of these.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_silu_bwd_matches_finite_differences(oracle):
    rng = np.random.default_rng(11)
    M, I = 64, 256
    g = f64(bf16(rng.standard_normal((M, I)) * 3.0))
    u = f64(bf16(rng.standard_normal((M, I)) * 2.0))
    dh = f64(bf16(rng.standard_normal((M, I)) * 1e-2))
    gu = np.concatenate([bf16(g), bf16(u)], axis=1)
    dgu, alt, _ = oracle.silu_mul_bwd(gu, bf16(dh))
    dg, du = f64(dgu[:, :I]), f64(dgu[:, I:])

    def fwd(gv, uv):   # h = silu(g) * u, binary64, independent of the oracle
        return gv * expit(gv) * uv

    eps = 1e-6
    dg_fd = dh * (fwd(g + eps, u) - fwd(g - eps, u)) / (2 * eps)
    du_fd = dh * (fwd(g, u + eps) - fwd(g, u - eps)) / (2 * eps)
    # BF16 rounding (2^-9 relative) plus the finite-difference error
    assert np.all(np.abs(dg - dg_fd) <= 2.0 ** -8 * np.abs(dg_fd) + 1e-9)
    assert np.all(np.abs(du - du_fd) <= 2.0 ** -8 * np.abs(du_fd) + 1e-9)
    # the analytic value rounds to the oracle's BF16 (or, at a midpoint, to its neighbour)
    s = expit(g)
    exact_dg = dh * u * s * (1 + g * (1 - s))
    rb = bf16(exact_dg)
    assert np.all((rb == dgu[:, :I]) | (rb == alt[:, :I]))


def test_silu_bwd_closed_forms(oracle):
    I = 128
    g = np.zeros((2, I))
    g[1] = 30.0                     # sigmoid(30) = 1 - 9.4e-14: silu ~ g, silu' ~ 1
    u = np.full((2, I), 0.75)
    dh = np.full((2, I), 0.5)
    gu = np.concatenate([bf16(g), bf16(u)], axis=1)
    dgu, _, _ = oracle.silu_mul_bwd(gu, bf16(dh))
    # g = 0: sigmoid = 1/2, silu = 0, silu' = 1/2 -> dg = dh*u/2 = 0.1875 (exact), du = 0
    assert np.all(f64(dgu[0, :I]) == 0.1875)
    assert np.all(f64(dgu[0, I:]) == 0.0)
    # g = 30: dg -> dh*u = 0.375, du -> dh*g = 15 (both exact BF16 after rounding)
    assert np.all(f64(dgu[1, :I]) == 0.375)
    assert np.all(f64(dgu[1, I:]) == 15.0)


def test_silu_bwd_quant_is_the_gradient_quantizer(oracle):
    rng = np.random.default_rng(12)
    M, I = 128, 256
    gu = bf16(rng.standard_normal((M, 2 * I)) * 2.0)
    dh = bf16(rng.standard_normal((M, I)) * 1e-3)
    q, s, qT, sT, dgu, _ = oracle.silu_mul_bwd_quant(gu, dh)
    q2, s2 = oracle.quantize_1x128(dgu)
    qT2, sT2 = oracle.quantize_128x1(dgu)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    assert np.array_equal(qT, qT2) and np.array_equal(sT, sT2)
    assert q.shape == (M, 2 * I) and qT.shape == (2 * I, M)


def _rms_fwd(x, gamma, eps):
    """y = (x * r) * gamma with r from x, binary64 (no BF16 rounding), numpy only."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)
    return x * r * gamma[None, :]


def test_rmsnorm_bwd_matches_finite_differences(oracle):
    rng = np.random.default_rng(13)
    M, K, eps = 8, 256, 1e-5
    x = f64(bf16(rng.standard_normal((M, K)) * 1.5))
    gamma = f64(bf16(1.0 + 0.1 * rng.standard_normal(K)))
    dy = f64(bf16(rng.standard_normal((M, K)) * 1e-2))
    rstd = (1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)).astype(np.float32)
    dx, mag, dgamma = oracle.rmsnorm_bwd(bf16(x), bf16(gamma), rstd, bf16(dy))
    # d/dx of L = sum(dy * y(x)) by central differences, one coordinate at a time
    h = 1e-6
    fd = np.zeros((M, K))
    for j in range(K):
        xp, xm = x.copy(), x.copy()
        xp[:, j] += h
        xm[:, j] -= h
        fd[:, j] = np.sum(dy * (_rms_fwd(xp, gamma, eps) - _rms_fwd(xm, gamma, eps)), axis=1) / (2 * h)
    got = f64(dx)
    assert np.all(np.abs(got - fd) <= 2.0 ** -8 * mag + 1e-10), float(np.max(np.abs(got - fd) / (mag + 1e-30)))
    # dgamma = sum over rows of dy * x * r, against a numpy reduction
    ref = np.sum(dy * x * rstd.astype(np.float64)[:, None], axis=0)
    assert np.allclose(dgamma, ref, rtol=1e-12, atol=1e-18)


def test_rmsnorm_bwd_special_rows(oracle):
    K, eps = 128, 1e-5
    x = np.zeros((3, K))
    x[0] = 2.0                      # constant row
    x[2, ::2] = 1.0                 # half-zero row
    x[2, 1::2] = -1.0
    gamma = np.ones(K)
    dy = np.zeros((3, K))
    dy[0] = 0.25
    dy[1] = 0.5                     # a zero row of x: dx = r * gamma * dy exactly
    dy[2] = 1.0
    rstd = (1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)).astype(np.float32)
    dx, _, _ = oracle.rmsnorm_bwd(bf16(x), bf16(gamma), rstd, bf16(dy))
    r = rstd.astype(np.float64)
    # constant row c with constant dy d: dx = r d (1 - r^2 c^2) = r d eps / (c^2 + eps)
    expect0 = r[0] * 0.25 * (1.0 - r[0] ** 2 * 4.0)
    assert np.all(f64(dx[0]) == f64(bf16(np.full(K, expect0))))
    assert np.all(f64(dx[1]) == f64(bf16(np.full(K, r[1] * 0.5))))
    # +-1 row with dy = 1: S = sum(x) = 0, so dx = r * dy
    assert np.all(f64(dx[2]) == f64(bf16(np.full(K, r[2]))))


def test_requant_128x1_is_the_128x1_quantization_of_the_dequantized_values(oracle):
    """The WGrad operand from the saved FP8: decode(q)*s in binary32 (numpy), rounded to
    BF16 (torch), then the 128x1 quantization of those values (numpy's binary32 division
    and torch's E4M3 cast for the codes)."""
    rng = np.random.default_rng(14)
    M, K = 256, 384
    x = rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, (1, K)))
    q, s = oracle.quantize_1x128(bf16(x))
    qT, sT = oracle.requant_128x1(q, s)
    xhat = (oracle.e4m3_decode(q).astype(np.float32) *
            np.repeat(s.T, 128, axis=1).astype(np.float32))          # [M, K] binary32
    assert xhat.dtype == np.float32
    xhat = torch.from_numpy(xhat).to(torch.bfloat16).to(torch.float32).numpy()   # BF16 RNE
    g = xhat.reshape(M // 128, 128, K)
    amax = np.abs(g).max(axis=1)                                     # [M/128, K]
    s_ref = amax / np.float32(448.0)
    assert np.array_equal(sT.view(np.uint32), s_ref.view(np.uint32))
    v = np.clip(g / s_ref[:, None, :], -448.0, 448.0)                # binary32 division
    codes = torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = codes.transpose(2, 0, 1).reshape(K, M)                     # qT[k, m]
    assert np.array_equal(qT, ref)
    # a group whose values are exactly E4M3 grid points times a power of two is unchanged
    # by the round trip: requantizing the exactly representable 1x128 groups of the
    # transpose returns the same codes
    z = np.zeros((128, 128))
    z[:, 0] = 448.0 * 2.0 ** -3
    z[5, 1] = -3.0
    qz, sz = oracle.quantize_1x128(bf16(z))
    qTz, sTz = oracle.requant_128x1(qz, sz)
    assert sTz[0, 0] == np.float32(2.0 ** -3) and np.all(qTz[0] == 0x7E)
