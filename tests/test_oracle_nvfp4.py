"""Pins of the oracle's NVFP4 routines (the rollout format the QeRL page names).

Format: FP4 E2M1 elements, 16 per E4M3 block scale, a per-row FP32 scale on top; the
library's reading of the recipe is g = fl32(amax/2688), sb = E4M3(fl32(bmax/fl32(6g))),
code = E2M1(fl32(x / fl32(decode(sb) g))).  Checks that do not reuse the oracle's code:
  * the E2M1 encoder against a brute-force nearest search over the 8 magnitudes, ties to
    the even mantissa bit (the even code), on a dense grid, every tie and random values;
  * exactly representable rows (grid values times exact block scales times 2^e, one
    element at 6 * 448 * 2^e) come back as the same codes, block scales and 2^e, and
    dequantize to themselves;
  * exact ties of the quotient with non-power-of-two block scales round to even;
  * scale invariance under powers of two;
  * every code is a nearest grid point given its block's scale, and every block scale is
    torch's E4M3 cast of the block's ratio;
  * the GEMM equals numpy's binary64 matmul of operands dequantized through the format's
    value table and torch's E4M3 decoding.
"""
import numpy as np
import torch

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])   # codes 0..7


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e4m3_cast(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def unpack(q: np.ndarray) -> np.ndarray:
    """[R, K/2] packed bytes -> [R, K] codes (element 2i in the low nibble)."""
    out = np.empty((q.shape[0], 2 * q.shape[1]), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def code_values(codes: np.ndarray) -> np.ndarray:
    v = E2M1_MAG[codes & 0x7]
    return np.where(codes & 0x8, -v, v)


def dequant(q, sf, g):
    """x^ from the format's value table and torch's E4M3 decoding (not the oracle's)."""
    c = code_values(unpack(q))
    s = np.repeat(e4m3_values(sf), 16, axis=1)
    return c * s * g.astype(np.float64)[:, None]


def brute_e2m1(v: np.ndarray) -> np.ndarray:
    out = np.empty(v.shape, dtype=np.uint8)
    for i, x in enumerate(v.astype(np.float64)):
        a = abs(x)
        if a >= 6.0:
            c = 7
        else:
            d = np.abs(E2M1_MAG - a)
            best = np.flatnonzero(d == d.min())
            c = int(best[0]) if best.size == 1 else int(best[best % 2 == 0][0])
        out[i] = c | (8 if np.signbit(x) else 0)
    return out


def test_e2m1_decode_is_the_format(oracle):
    vals = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(vals[:8], E2M1_MAG)
    assert np.array_equal(vals[8:], -E2M1_MAG)
    assert np.signbit(vals[8])


def test_e2m1_encoder_is_nearest_even(oracle):
    rng = np.random.default_rng(3)
    grid = np.arange(-640, 641, dtype=np.float64) / 64.0       # every tie, saturation
    mids = (E2M1_MAG[:-1] + E2M1_MAG[1:]) / 2.0
    ties = np.concatenate([mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 10)])
    rnd = rng.uniform(-9.0, 9.0, 4000)
    tiny = np.array([0.0, -0.0, 1e-30, -1e-30, 0.2499999, -0.25, 6.0, -6.0, 1e30, -1e30])
    v = np.concatenate([grid, ties, rnd, tiny]).astype(np.float32)
    assert np.array_equal(oracle.e2m1_encode(v), brute_e2m1(v))


def exact_rows(oracle, rng, M, K, exps):
    """Rows of grid values times exact block scales times 2^e (one element 6*448*2^e per
    row).  Returns (x float64 [M,K], codes [M,K], sf [M,K/16])."""
    nb = K // 16
    codes = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    sf = rng.integers(0x08, 0x7F, size=(M, nb)).astype(np.uint8)   # normal E4M3 scales
    for r in range(M):
        sf[r, rng.integers(0, nb)] = 0x7E                           # 448: the row maximum
        for b in range(nb):
            codes[r, 16 * b + rng.integers(0, 16)] = 0x7 | (rng.integers(0, 2) << 3)   # +-6
    x = code_values(codes) * np.repeat(e4m3_values(sf), 16, axis=1) * (2.0 ** exps)[:, None]
    return x, codes, sf


def test_nvfp4_exact_rows_identity(oracle):
    rng = np.random.default_rng(4)
    M, K = 8, 256
    exps = rng.integers(-40, 20, size=M).astype(np.float64)
    x, codes, sf = exact_rows(oracle, rng, M, K, exps)
    x[5] = 0.0                                   # all-zero row
    x[6, 32:48] = 0.0                            # all-zero block
    codes[5] = 0
    codes[6, 32:48] = np.where(np.signbit(x[6, 32:48]), 8, 0)
    xb = bf16_bits(x)
    assert np.array_equal(oracle.bf16_to_f32(xb).astype(np.float64), x)   # exact in BF16
    q, s, g = oracle.quantize_nvfp4(xb)
    assert q.shape == (M, K // 2) and s.shape == (M, K // 16) and g.shape == (M,)
    got = unpack(q)
    assert np.array_equal(got[[0, 1, 2, 3, 4, 7]], codes[[0, 1, 2, 3, 4, 7]])
    assert np.array_equal(got[6][codes[6] != 8], codes[6][codes[6] != 8])
    assert np.all(got[5] == 0) and np.all(got[6, 32:48] == 0) and np.all(s[5] == 0) and g[5] == 0.0
    assert s[6, 2] == 0
    keep = [0, 1, 2, 3, 4, 7]
    assert np.array_equal(s[keep], sf[keep])
    assert np.array_equal(g[keep], (2.0 ** exps[keep]).astype(np.float32))
    assert np.array_equal(dequant(q, s, g), x)


def test_nvfp4_quotient_ties_round_to_even(oracle):
    """Block scales 1.125, 1.375, 1.625, 1.875 (times 2^k): each element is a midpoint of
    the E2M1 grid times the block's decode scale, so x / d is an exact tie."""
    K = 128
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    want = np.array([0, 2, 2, 4, 4, 6, 6], dtype=np.uint8)   # the even neighbours
    sfc = np.array([0x39, 0x3B, 0x3D, 0x3F, 0x41, 0x4B, 0x55], dtype=np.uint8)
    rows, codes = [], []
    for e in (-7, 0, 9):
        x = np.zeros(K)
        c = np.zeros(K, dtype=np.uint8)
        x[0], c[0] = 6.0 * 448.0 * 2.0 ** e, 7                  # block 0: scale 448, g = 2^e
        for b, sc in enumerate(sfc, start=1):
            d = e4m3_values(np.array([sc]))[0] * 2.0 ** e
            x[16 * b], c[16 * b] = 6.0 * d, 7
            for i, (m, w) in enumerate(zip(mids, want)):
                sign = -1.0 if i % 2 else 1.0
                x[16 * b + 1 + i] = sign * m * d
                c[16 * b + 1 + i] = w | (8 if sign < 0 else 0)
        rows.append(x)
        codes.append(c)
    x = np.array(rows)
    xb = bf16_bits(x)
    assert np.array_equal(oracle.bf16_to_f32(xb).astype(np.float64), x)
    q, s, g = oracle.quantize_nvfp4(xb)
    got = unpack(q)
    want_codes = np.array(codes)
    nz = x != 0
    assert np.array_equal(got[nz], want_codes[nz])
    assert np.array_equal(s[:, 1:8], np.tile(sfc, (3, 1)))


def test_nvfp4_scale_invariance(oracle):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 512)) * 0.02
    x[:, 7] *= 40.0                                             # an outlier channel
    q0, s0, g0 = oracle.quantize_nvfp4(bf16_bits(x))
    for k in (-30, -3, 5, 60):
        q, s, g = oracle.quantize_nvfp4(bf16_bits(x * 2.0 ** k))
        assert np.array_equal(q, q0) and np.array_equal(s, s0)
        assert np.array_equal(g, (g0.astype(np.float64) * 2.0 ** k).astype(np.float32))


def test_nvfp4_codes_nearest_and_scales_are_e4m3_casts(oracle):
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal((6, 1024)) * 10.0 ** rng.uniform(-6, 3, (6, 1)),
                        rng.laplace(size=(2, 1024)) * 1e-3])
    x[7, 100] = 3.0                                             # one outlier: many tiny blocks
    xb = bf16_bits(x)
    xf = oracle.bf16_to_f32(xb).astype(np.float32)
    q, s, g = oracle.quantize_nvfp4(xb)
    bmax = np.abs(xf).reshape(8, -1, 16).max(axis=2)
    g6 = np.float32(6.0) * g
    assert np.array_equal(s, e4m3_cast(bmax / g6[:, None]))
    d = np.repeat((e4m3_values(s).astype(np.float32) * g[:, None]).astype(np.float64), 16, axis=1)
    xd = xf.astype(np.float64)
    err = np.abs(xd - code_values(unpack(q)) * d)
    best = np.min(np.abs(np.abs(xd)[..., None] - E2M1_MAG * d[..., None]), axis=-1)
    assert np.all(err <= best * (1 + 2.0 ** -20) + 1e-300)
    assert np.all(g == (np.abs(xf).max(axis=1) / np.float32(2688.0)))


def test_gemm_nvfp4_exact_operands(oracle):
    rng = np.random.default_rng(7)
    M, N, K = 5, 7, 256
    x, _, _ = exact_rows(oracle, rng, M, K, rng.integers(-8, 8, size=M).astype(np.float64))
    w, _, _ = exact_rows(oracle, rng, N, K, rng.integers(-8, 8, size=N).astype(np.float64))
    qx, sx, gx = oracle.quantize_nvfp4(bf16_bits(x))
    qw, sw, gw = oracle.quantize_nvfp4(bf16_bits(w))
    y = oracle.gemm_nvfp4(qx, sx, gx, qw, sw, gw)
    assert np.array_equal(y, x @ w.T)


def test_gemm_nvfp4_is_the_dequantized_matmul(oracle):
    rng = np.random.default_rng(8)
    M, N, K = 9, 24, 512
    x = rng.standard_normal((M, K))
    w = rng.standard_normal((N, K)) * 0.02
    qx, sx, gx = oracle.quantize_nvfp4(bf16_bits(x))
    qw, sw, gw = oracle.quantize_nvfp4(bf16_bits(w))
    y = oracle.gemm_nvfp4(qx, sx, gx, qw, sw, gw)
    ref = dequant(qx, sx, gx) @ dequant(qw, sw, gw).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    m = rng.integers(0, M, 50)
    n = rng.integers(0, N, 50)
    assert np.array_equal(oracle.gemm_nvfp4_sampled(qx, sx, gx, qw, sw, gw, m, n), y[m, n])


def test_e2m1_bits_range_matches_array_encoder(oracle):
    first = 0x3F000000
    codes = oracle.e2m1_encode_bits_range(first, 1 << 16)
    vals = np.arange(first, first + (1 << 16), dtype=np.uint32).view(np.float32)
    assert np.array_equal(codes, oracle.e2m1_encode(vals))
    assert np.array_equal(codes, brute_e2m1(vals))
