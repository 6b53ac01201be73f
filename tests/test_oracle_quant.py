"""Pins of the oracle's quantizers (1x128, 128x1 transposed, 128x128 blocks).

Scheme: "Technical summary: Jet-RL", section "Quantization Scheme" -- activations 1x128,
weights 128x128, WGrad operands 128x1; scale = fl32(amax/448) is this library's reading.
Checks that do not reuse the oracle's formula:
  * exactly representable groups (E4M3 grid points times 2^j with the group maximum
    448*2^j) must give s = 2^j and codes equal to the grid points' codes (identity);
    different j per group pins the scale layout and the transposition,
  * scale invariance under powers of two,
  * round-trip error bounds of E4M3 and the amax element landing on 448*s,
  * an all-zero group, and a denormal-amax group that drives the quantizer into
    saturation.
"""
import numpy as np
import torch

POS_CODES = np.array([c for c in range(1, 0x7F)], dtype=np.uint8)  # finite, non-zero


def grid_values(oracle):
    return oracle.e4m3_decode(POS_CODES)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_group(oracle, rng, j, n=128):
    """n values on the E4M3 grid (random codes and signs) times 2^j, with one element
    exactly 448*2^j.  Returns (values, codes)."""
    codes = rng.choice(POS_CODES, size=n)
    codes[rng.integers(0, n)] = 0x7E
    signs = rng.integers(0, 2, size=n).astype(np.uint8) << 7
    codes = codes | signs
    vals = oracle.e4m3_decode(codes) * 2.0 ** j
    return vals, codes


def test_exact_1x128_rows_identity_and_scale_layout(oracle):
    rng = np.random.default_rng(0)
    R, C = 6, 384
    x = np.zeros((R, C))
    codes = np.zeros((R, C), dtype=np.uint8)
    js = rng.integers(-20, 20, size=(R, C // 128))
    for r in range(R):
        for b in range(C // 128):
            v, c = exact_group(oracle, rng, js[r, b])
            x[r, b * 128:(b + 1) * 128] = v
            codes[r, b * 128:(b + 1) * 128] = c
    xb = bf16_bits(x)
    assert np.array_equal(oracle.bf16_to_f32(xb).astype(np.float64), x)  # exact in BF16
    q, s = oracle.quantize_1x128(xb)
    assert np.array_equal(q, codes)
    assert s.shape == (C // 128, R)
    assert np.array_equal(s, (2.0 ** js.T).astype(np.float32))


def test_exact_128x1_is_transposed_and_per_column(oracle):
    rng = np.random.default_rng(1)
    M, K = 256, 5
    x = np.zeros((M, K))
    codes = np.zeros((M, K), dtype=np.uint8)
    js = rng.integers(-10, 10, size=(M // 128, K))
    for b in range(M // 128):
        for k in range(K):
            v, c = exact_group(oracle, rng, js[b, k])
            x[b * 128:(b + 1) * 128, k] = v
            codes[b * 128:(b + 1) * 128, k] = c
    Kp = 128  # the quantizer wants K % 128 == 0 only for 1x128; pad columns with zeros
    xp = np.zeros((M, Kp))
    xp[:, :K] = x
    qT, sT = oracle.quantize_128x1(bf16_bits(xp))
    assert qT.shape == (Kp, M) and sT.shape == (M // 128, Kp)
    assert np.array_equal(qT[:K], codes.T)
    assert np.array_equal(sT[:, :K], (2.0 ** js).astype(np.float32))
    assert np.all(qT[K:] == 0) and np.all(sT[:, K:] == 0)


def test_exact_128x128_single_scale_per_block(oracle):
    rng = np.random.default_rng(2)
    N, K = 256, 384
    w = np.zeros((N, K))
    codes = np.zeros((N, K), dtype=np.uint8)
    js = rng.integers(-12, 4, size=(N // 128, K // 128))
    for bn in range(N // 128):
        for bk in range(K // 128):
            v, c = exact_group(oracle, rng, js[bn, bk], n=128 * 128)
            w[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128] = v.reshape(128, 128)
            codes[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128] = c.reshape(128, 128)
    q, s, qT = oracle.quantize_128x128(bf16_bits(w))
    assert np.array_equal(q, codes)
    assert np.array_equal(qT, codes.T)
    assert np.array_equal(s, (2.0 ** js).astype(np.float32))


def test_block_scale_is_shared_by_the_whole_block(oracle):
    """One large element sets the scale of all 128x128 entries, not just its row."""
    w = np.full((128, 128), 1.0)
    w[5, 7] = 448.0 * 64
    q, s, _ = oracle.quantize_128x128(bf16_bits(w))
    assert s[0, 0] == 64.0
    assert q[5, 7] == 0x7E
    # 1.0 / 64 = 2^-6 is the smallest normal E4M3 value (code 0x08)
    assert np.all(q[np.arange(128) != 5] == 0x08)


def test_scale_invariance(oracle):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    xb = bf16_bits(x)
    xf = oracle.bf16_to_f32(xb)
    q0, s0 = oracle.quantize_1x128(xb)
    for j in (-12, -3, 5, 17):
        xj = bf16_bits(xf * np.float32(2.0 ** j))  # exact: power-of-two scaling of BF16
        q, s = oracle.quantize_1x128(xj)
        assert np.array_equal(q, q0)
        assert np.array_equal(s, s0 * np.float32(2.0 ** j))


def test_round_trip_bounds(oracle):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((128, 1024)) * np.exp(rng.uniform(-6, 6, (128, 1)))).astype(np.float32)
    xb = bf16_bits(x)
    xf = oracle.bf16_to_f32(xb).astype(np.float64)
    q, s = oracle.quantize_1x128(xb)
    srow = np.repeat(s.T.astype(np.float64), 128, axis=1)      # [R, C]
    deq = oracle.e4m3_decode(q) * srow
    err = np.abs(xf - deq)
    normal = np.abs(xf) >= srow * 2.0 ** -6
    # half an E4M3 step (relative 2^-4 in the normal range, 2^-10*s below it), plus the
    # binary32 rounding of the quotient
    assert np.all(err[normal] <= np.abs(xf[normal]) * (2.0 ** -4) * (1 + 2.0 ** -20))
    assert np.all(err[~normal] <= srow[~normal] * 2.0 ** -10 * (1 + 2.0 ** -20))
    # the group maximum lands on 448*s up to the rounding of s
    amax = np.abs(xf).reshape(128, 8, 128).max(axis=2)
    code_at_max = np.abs(oracle.e4m3_decode(q)).reshape(128, 8, 128).max(axis=2)
    assert np.all(code_at_max == 448.0)
    assert np.all(np.abs(448.0 * s.T - amax) <= amax * 2.0 ** -23)


def test_zero_group_and_denormal_amax(oracle):
    x = np.zeros((2, 256), dtype=np.float32)
    x[1, 128] = 2.0 ** -130          # a BF16 subnormal; s = fl32(2^-130/448) loses bits
    x[1, 129] = -(2.0 ** -131)
    q, s = oracle.quantize_1x128(bf16_bits(x))
    assert s[0, 0] == 0 and s[1, 0] == 0 and s[0, 1] == 0
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0)
    assert s[1, 1] > 0
    # 2^-130 / s exceeds 448 because s was rounded down in the subnormal range
    assert np.float64(2.0 ** -130) / np.float64(s[1, 1]) > 448.0
    assert q[1, 128] == 0x7E
    quotient = np.float32(-(2.0 ** -131)) / s[1, 1]          # IEEE binary32 division
    assert q[1, 129] == oracle.e4m3_encode(np.array([quotient], np.float32))[0]
    assert np.all(q[1, 130:] == 0)


def test_quotient_is_the_ieee_binary32_division_in_the_normal_range(oracle):
    """Every code is the E4M3 rounding of the correctly rounded binary32 quotient x / s,
    not of x times a rounded reciprocal: random groups whose maxima are not powers of two
    (so s is not one either), spread over 2^-20 .. 2^20.  The reference is numpy's IEEE
    binary32 division and torch's float8_e4m3fn cast, two routines the oracle does not use."""
    rng = np.random.default_rng(5)
    R, C = 256, 1024
    sig = 2.0 ** rng.uniform(-20, 20, size=(R, 1))
    x = (rng.standard_normal((R, C)) * sig).astype(np.float32)
    xb = bf16_bits(x)
    xf = oracle.bf16_to_f32(xb).astype(np.float32)
    q, s = oracle.quantize_1x128(xb)
    g = xf.reshape(R, C // 128, 128)
    amax = np.abs(g).max(axis=2)
    s_ref = amax / np.float32(448.0)                      # binary32 division
    assert s_ref.dtype == np.float32
    assert np.array_equal(s.T.view(np.uint32), s_ref.view(np.uint32))
    # almost no scale is a power of two, so a reciprocal product differs somewhere
    mant = s_ref.view(np.uint32) & 0x7FFFFF
    assert np.mean(mant != 0) > 0.99
    v = g / s_ref[:, :, None]                             # binary32 division, per element
    assert v.dtype == np.float32
    v = np.clip(v, -448.0, 448.0).reshape(R, C)
    ref = torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = q != ref
    assert not bad.any(), f"{int(bad.sum())} codes differ, first at {np.argwhere(bad)[0]}"
    # the reciprocal form really differs on these inputs (so this test can tell them apart)
    v_rcp = np.clip((g * (np.float32(1.0) / s_ref)[:, :, None]).reshape(R, C), -448.0, 448.0)
    rcp = torch.from_numpy(np.ascontiguousarray(v_rcp)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (rcp != ref).any()
