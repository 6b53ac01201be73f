"""Pins of the oracle's number formats (E4M3 encode/decode, BF16 rounding).

The Jet-RL technical summary ("Quantization Scheme") says only "FP8"; the oracle reads it
as OCP E4M3 "FN" (bias 7, max 448, no infinities, S.1111.111 = NaN).  These tests pin the
oracle's encoder and decoder against sources that share none of its code:
  * closed-form values of the format (powers of two and the limits it names),
  * torch's own float8_e4m3fn decoder and encoder (a library routine),
  * a brute-force nearest-value search over the 254 finite codes (written here),
so that a slip in the oracle's exponent, rounding, tie, subnormal or sign handling fails.
"""
import numpy as np
import pytest
import torch


def all_codes_torch():
    b = torch.arange(256, dtype=torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_for_every_code(oracle):
    mine = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = all_codes_torch()
    nan_mine = np.isnan(mine)
    assert np.array_equal(nan_mine, np.isnan(ref))
    assert set(np.nonzero(nan_mine)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan_mine], ref[~nan_mine])
    assert np.array_equal(np.signbit(mine[~nan_mine]), np.signbit(ref[~nan_mine]))


# Closed forms of the E4M3 format's named values (OCP OFP8 v1.0: zero, subnormals with
# spacing 2^-9, min normal 2^-6, exponent bias 7, max normal 1.75 * 2^8, NaN S.1111.111).
NAMED = [(0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
         (0x08, 2.0 ** -6), (0x38, 1.0), (0x7E, 448.0), (0xFE, -448.0),
         (0x40, 2.0), (0x3C, 1.5), (0x30, 0.5)]


@pytest.mark.parametrize("code,value", NAMED)
def test_named_values(oracle, code, value):
    d = oracle.e4m3_decode(np.array([code], dtype=np.uint8))[0]
    assert d == value and np.signbit(d) == np.signbit(value)
    assert oracle.e4m3_encode(np.array([value], dtype=np.float32))[0] == code


def test_encode_inverts_decode(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def brute_force_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by search over the code table; ties to the even code;
    saturating at +-448; the sign of the input is kept (also for results of zero)."""
    codes = np.arange(0, 0x7F, dtype=np.int64)                    # 0x00 .. 0x7E, ascending
    vals = all_codes_torch()[:0x7F]
    assert np.all(np.diff(vals) > 0)
    a = np.abs(v.astype(np.float64))
    i = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, len(vals) - 1)
    j = np.clip(i + 1, 0, len(vals) - 1)
    dlo = a - vals[i]
    dhi = vals[j] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[j] % 2 == 0) & (j != i))
    idx = np.where(pick_hi, j, i)
    idx = np.where(a >= 448.0, len(vals) - 1, idx)
    out = codes[idx].astype(np.uint8)
    return out | (np.signbit(v).astype(np.uint8) << 7)


def test_encode_exhaustive_band_vs_brute_force_and_torch(oracle):
    """Every binary32 pattern with magnitude in [2^-11, 2^9): all rounding decisions,
    ties, binade edges, subnormals and saturation lie inside this band."""
    first = np.float32(2.0 ** -11).view(np.uint32).item()
    last = np.float32(2.0 ** 9).view(np.uint32).item()
    chunk = 1 << 24
    for start in range(first, last, chunk):
        n = min(chunk, last - start)
        mine = oracle.e4m3_encode_bits_range(start, n)
        v = np.arange(start, start + n, dtype=np.uint32).view(np.float32)
        assert np.array_equal(mine, brute_force_encode(v)), f"chunk at {start:#x}"
        tv = torch.from_numpy(np.clip(v, -448.0, 448.0))
        ref = tv.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(mine, ref), f"torch chunk at {start:#x}"


def test_encode_random_full_range(oracle):
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    mine = oracle.e4m3_encode(v)
    assert np.array_equal(mine, brute_force_encode(v))
    ref = torch.from_numpy(np.clip(v, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(mine, ref.numpy())


def test_saturation_and_signed_zero(oracle):
    v = np.array([448.0, 463.99, 464.0, 1000.0, 3.0e38, -448.0, -463.99, -464.0, -1000.0,
                  -3.0e38], dtype=np.float32)
    assert oracle.e4m3_encode(v).tolist() == [0x7E] * 5 + [0xFE] * 5
    z = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, -(2.0 ** -10)], dtype=np.float32)
    # 2^-10 is the tie between 0 and 2^-9: ties go to the even code, 0
    assert oracle.e4m3_encode(z).tolist() == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]


def test_sign_symmetry(oracle):
    rng = np.random.default_rng(7)
    v = np.abs(rng.standard_normal(1 << 16) * 30).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(-v), oracle.e4m3_encode(v) | 0x80)


def test_bf16_rounding_matches_torch(oracle):
    rng = np.random.default_rng(99)
    bits = rng.integers(0, 2 ** 32, size=1 << 14, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 3.0e38)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = oracle.f64_to_bf16(v.astype(np.float64))
    assert np.array_equal(mine, ref)
    # ties: values exactly halfway between two BF16 neighbours go to the even one
    t = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], dtype=np.float64)
    assert oracle.f64_to_bf16(t).tolist() == [0x3F80, 0x3F82, 0xBF80]
