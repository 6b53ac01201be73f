"""Pins of the oracle's fused producers: RMSNorm -> quantize and SiLU-mul -> quantize.

"Technical summary: Jet-RL", section "Implementation": fused activation and RMSNorm
kernels feed the quantizer; section "Quantization Scheme": the saved activation is FP8,
produced by the preceding operator.  The RMSNorm and SiLU formulas are the textbook ones
(the pages print none).  Independent checks:
  * RMSNorm closed forms: a constant row normalises to +-1 (codes 0x7E/0xFE, s = 1/448);
    a zero row gives zero codes and s = 0; eps = 0 makes y invariant under x -> 2^j x;
    power-of-two gamma multiplies y exactly (pins gamma's column index);
    rstd agrees with numpy's binary64 formula to 2 binary32 ulps (four single-precision
    roundings: the mean, + eps, the square root and the division);
  * SiLU-mul against scipy's logistic function in binary64 (a library routine), the zero
    cases, the large-gate limit silu(g) ~ g, and the gate/up column order.
"""
import numpy as np
import pytest
import torch


def bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


ONE_BF16 = 0x3F80


def test_rmsnorm_constant_and_zero_rows(oracle):
    K = 256
    x = np.zeros((128, K), dtype=np.float32)
    x[0] = 3.0
    x[1] = -0.75
    x[2] = 1e4
    gamma = bf16_bits(np.ones(K))
    q, s, qT, sT, rstd, y = oracle.rmsnorm_quant(bf16_bits(x), gamma, 1e-5)
    assert np.all(y[0] == ONE_BF16) and np.all(y[2] == ONE_BF16)
    assert np.all(y[1] == (ONE_BF16 | 0x8000))
    for r in (0, 1, 2):
        assert np.all(s[:, r] == np.float32(1.0) / np.float32(448.0))
        assert np.all(q[r] == (0x7E if x[r, 0] > 0 else 0xFE))
    assert np.all(y[3:] == 0) and np.all(q[3:] == 0) and np.all(s[:, 3:] == 0)
    assert rstd[3] == np.float32(1.0) / np.sqrt(np.float32(1e-5))


def test_rmsnorm_scale_invariance_with_zero_eps(oracle):
    rng = np.random.default_rng(40)
    x = rng.standard_normal((128, 512)).astype(np.float32)
    g = bf16_bits(1.0 + 0.1 * rng.standard_normal(512))
    xb = bf16_bits(x)
    y0, r0 = oracle.rmsnorm(xb, g, 0.0)
    xf = oracle.bf16_to_f32(xb)
    for j in (-20, 7):
        y, r = oracle.rmsnorm(bf16_bits(xf * np.float32(2.0 ** j)), g, 0.0)
        assert np.array_equal(y, y0)
        assert np.array_equal(r, r0 * np.float32(2.0 ** -j))


def test_rmsnorm_gamma_is_per_column(oracle):
    K = 384
    x = np.ones((4, K), dtype=np.float32)
    gamma_vals = 2.0 ** (np.arange(K) % 5)
    y, r = oracle.rmsnorm(bf16_bits(x), bf16_bits(gamma_vals), 1e-5)
    y1, _ = oracle.rmsnorm(bf16_bits(x), bf16_bits(np.ones(K)), 1e-5)
    base = oracle.bf16_to_f32(y1).astype(np.float64)
    assert np.array_equal(oracle.bf16_to_f32(y).astype(np.float64), base * gamma_vals[None, :])


def test_rmsnorm_rstd_vs_binary64_formula(oracle):
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((300, 640)) * np.exp(rng.uniform(-4, 4, (300, 1)))).astype(np.float32)
    xb = bf16_bits(x)
    xf = oracle.bf16_to_f32(xb).astype(np.float64)
    _, r = oracle.rmsnorm(xb, bf16_bits(np.ones(640)), 1e-5)
    ref = 1.0 / np.sqrt(np.mean(xf * xf, axis=1) + 1e-5)
    ulp = np.spacing(r.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(r.astype(np.float64) - ref) <= 2 * ulp)


def test_silu_mul_vs_scipy_logistic(oracle):
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(42)
    M, I = 64, 256
    g = (rng.standard_normal((M, I)) * 3).astype(np.float32)
    u = rng.standard_normal((M, I)).astype(np.float32)
    gu = bf16_bits(np.concatenate([g, u], axis=1))
    h, alt, nflag = oracle.silu_mul(gu)
    gf = oracle.bf16_to_f32(gu[:, :I]).astype(np.float64)
    uf = oracle.bf16_to_f32(gu[:, I:]).astype(np.float64)
    ref = gf * special.expit(gf) * uf
    ref_bits = bf16_bits(ref.astype(np.float32))   # float32 then BF16: fine away from ties
    same = h == ref_bits
    flagged = h != alt
    assert np.all(same | flagged)
    assert nflag == int(flagged.sum())
    # the alternative is always the other BF16 neighbour
    hv = oracle.bf16_to_f32(h[flagged]).astype(np.float64)
    av = oracle.bf16_to_f32(alt[flagged]).astype(np.float64)
    gap = np.abs(hv - av) / np.maximum(np.abs(hv), np.abs(av))
    assert np.all((gap > 0) & (gap <= 2.0 ** -7))   # one BF16 step (8 significant bits)


def test_silu_mul_special_cases_and_gate_order(oracle):
    I = 128
    g = np.zeros((3, I), dtype=np.float32)
    u = np.ones((3, I), dtype=np.float32)
    g[1] = 30.0            # silu(30) = 30 / (1 + e^-30): rounds to 30 in BF16
    u[2] = 0.0
    g[2] = 5.0
    h, _, _ = oracle.silu_mul(bf16_bits(np.concatenate([g, u], axis=1)))
    hf = oracle.bf16_to_f32(h)
    assert np.all(hf[0] == 0.0) and np.all(hf[2] == 0.0)
    assert np.all(hf[1] == 30.0)
    # swapping gate and up changes the result: g = 30, u = 1  vs  g = 1, u = 30
    h2, _, _ = oracle.silu_mul(bf16_bits(np.concatenate([u[1:2], g[1:2]], axis=1)))
    assert np.all(oracle.bf16_to_f32(h2) != 30.0)
