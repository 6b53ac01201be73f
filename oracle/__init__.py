"""CPU oracle for the unified-precision FP8 linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import this package.  The product path (``block_scaled_fp8_x1_gb300``) never
imports, links or calls it, and it never calls the product path: the two share no code.

The arithmetic lives in plain C (``fp8rl_oracle.c``, compiled here with gcc,
``-ffp-contract=off``); this module only marshals numpy arrays.  What each routine computes,
and which passage of "Technical summary: Jet-RL" (section "Quantization Scheme") it
follows, is written beside the C code.

Array conventions (all numpy, C-contiguous):
  * BF16 tensors travel as ``uint16`` bit patterns.
  * E4M3 codes are ``uint8``; scales are ``float32``.
  * NVFP4 (E2M1) codes are packed two to a ``uint8``, element 2i in the low nibble; their
    E4M3 block scales are ``uint8`` [rows, K/16], the per-row scales ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8rl_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``fp8rl_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        sig = {
            "orc_set_threads": (None, [ctypes.c_int]),
            "orc_get_threads": (ctypes.c_int, []),
            "orc_have_openmp": (ctypes.c_int, []),
            "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_e4m3_encode_array": (None, [P, P, I64]),
            "orc_e4m3_encode_bits_range": (None, [ctypes.c_uint32, I64, P]),
            "orc_quant_group_f32": (None, [P, I64, P, P]),
            "orc_quantize_1x128": (None, [P, I64, I64, I64, P, I64, P]),
            "orc_quantize_128x1": (None, [P, I64, I64, I64, P, I64, P]),
            "orc_quantize_128x128": (None, [P, I64, I64, I64, P, I64, P, P]),
            "orc_rmsnorm": (None, [P, P, ctypes.c_float, I64, I64, P, P, P]),
            "orc_silu_mul": (I64, [P, I64, I64, P, P]),
            "orc_silu_mul_bwd": (I64, [P, P, I64, I64, P, P]),
            "orc_requant_128x1": (None, [P, P, I64, I64, P, P]),
            "orc_rmsnorm_bwd": (None, [P, P, P, P, I64, I64, P, P, P]),
            "orc_gemm": (None, [P, I64, P, I64, P, I64, P, I64, I64, I64, I64, I64, I64, P]),
            "orc_gemm_sampled": (None, [P, I64, P, I64, P, I64, P, I64, I64, I64, I64, P, P,
                                        I64, P]),
            "orc_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_e2m1_encode_array": (None, [P, P, I64]),
            "orc_e2m1_encode_bits_range": (None, [ctypes.c_uint32, I64, P]),
            "orc_quantize_nvfp4": (None, [P, I64, I64, I64, P, P, P]),
            "orc_gemm_nvfp4": (None, [P, P, P, I64, P, P, P, I64, I64, P]),
            "orc_gemm_nvfp4_sampled": (None, [P, P, P, P, P, P, I64, P, P, I64, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        lib.orc_set_threads(os.cpu_count() or 1)
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def threads() -> int:
    lib = _load()
    return lib.orc_get_threads() if lib.orc_have_openmp() else 1


# ------------------------------------------------------------------ scalar formats

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 (exact: the bits are the top half)."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round binary64 values to BF16 (nearest, ties to even); returns uint16 bits."""
    lib = _load()
    flat = np.asarray(v, dtype=np.float64).ravel()
    out = np.fromiter((lib.orc_f64_to_bf16(float(x)) for x in flat), dtype=np.uint16,
                      count=flat.size)
    return out.reshape(np.shape(v))


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes -> binary64 values (NaN for 0x7F/0xFF)."""
    lib = _load()
    table = np.array([lib.orc_e4m3_decode(b) for b in range(256)], dtype=np.float64)
    return table[_c(codes, np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Finite binary32 values -> E4M3 codes (RNE, saturating at +-448)."""
    x = _c(v, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


def e4m3_encode_bits_range(first: int, count: int) -> np.ndarray:
    """Codes for every binary32 bit pattern first, first+1, ..., first+count-1."""
    out = np.empty(count, dtype=np.uint8)
    _load().orc_e4m3_encode_bits_range(first, count, _p(out))
    return out


# ------------------------------------------------------------------ quantizers

def quant_group(x: np.ndarray):
    """One group of binary32 values -> (codes, scale)."""
    v = _c(x, np.float32).ravel()
    q = np.empty(v.size, dtype=np.uint8)
    s = np.empty(1, dtype=np.float32)
    _load().orc_quant_group_f32(_p(v), v.size, _p(q), _p(s))
    return q, s[0]


def quantize_1x128(a_bf16: np.ndarray):
    """A[R,C] (uint16 BF16 bits) -> q[R,C] uint8, s[C/128, R] float32."""
    a = _c(a_bf16, np.uint16)
    R, C = a.shape
    assert C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((C // 128, R), dtype=np.float32)
    _load().orc_quantize_1x128(_p(a), R, C, C, _p(q), C, _p(s))
    return q, s


def quantize_128x1(x_bf16: np.ndarray):
    """X[M,K] -> transposed codes qT[K,M] uint8, sT[M/128, K] float32."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert M % 128 == 0
    qT = np.empty((K, M), dtype=np.uint8)
    sT = np.empty((M // 128, K), dtype=np.float32)
    _load().orc_quantize_128x1(_p(x), M, K, K, _p(qT), M, _p(sT))
    return qT, sT


def quantize_128x128(w_bf16: np.ndarray, with_transpose: bool = True):
    """W[N,K] -> q[N,K], s[N/128, K/128], and qT[K,N] (or None)."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N // 128, K // 128), dtype=np.float32)
    qT = np.empty((K, N), dtype=np.uint8) if with_transpose else None
    _load().orc_quantize_128x128(_p(w), N, K, K, _p(q), K, _p(s),
                                 _p(qT) if qT is not None else None)
    return q, s, qT


def rmsnorm(x_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float, rstd_in=None):
    """y = bf16((x*rstd)*gamma); returns (y uint16 [M,K], rstd float32 [M])."""
    x = _c(x_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    M, K = x.shape
    y = np.empty((M, K), dtype=np.uint16)
    r = np.empty(M, dtype=np.float32)
    rin = _c(rstd_in, np.float32) if rstd_in is not None else None
    _load().orc_rmsnorm(_p(x), _p(g), ctypes.c_float(eps), M, K, _p(y), _p(r),
                        _p(rin) if rin is not None else None)
    return y, r


def silu_mul(gu_bf16: np.ndarray):
    """GU[M, 2I] -> (h uint16 [M,I], alt uint16 [M,I], n_flagged).

    ``alt`` differs from ``h`` only where the binary64 value lies within 2^-16 relative of a
    BF16 rounding midpoint; there it holds the other BF16 neighbour."""
    gu = _c(gu_bf16, np.uint16)
    M, I2 = gu.shape
    assert I2 % 2 == 0
    I = I2 // 2
    h = np.empty((M, I), dtype=np.uint16)
    alt = np.empty((M, I), dtype=np.uint16)
    n = _load().orc_silu_mul(_p(gu), M, I, _p(h), _p(alt))
    return h, alt, int(n)


def requant_128x1(q: np.ndarray, s: np.ndarray):
    """From X's 1x128 codes q[M,K] and scales s[K/128,M]: the 128x1 quantization of the
    dequantized BF16 values bf16(fl32(decode(q)*s)), transposed: (qT uint8 [K,M],
    sT float32 [M/128,K])."""
    qq = _c(q, np.uint8)
    ss = _c(s, np.float32)
    M, K = qq.shape
    assert M % 128 == 0 and K % 128 == 0 and ss.shape == (K // 128, M)
    qT = np.empty((K, M), dtype=np.uint8)
    sT = np.empty((M // 128, K), dtype=np.float32)
    _load().orc_requant_128x1(_p(qq), _p(ss), M, K, _p(qT), _p(sT))
    return qT, sT


def silu_mul_bwd(gu_bf16: np.ndarray, dh_bf16: np.ndarray):
    """SiLU-mul backward: GU[M, 2I] (the forward's gate | up) and dH[M, I] ->
    (dGU uint16 [M, 2I] = [dg | du] as BF16, alt uint16 [M, 2I], n_flagged).

    ``alt`` differs from ``dGU`` only where the binary64 value lies within 2^-16 relative of
    a BF16 rounding midpoint; there it holds the other BF16 neighbour."""
    gu = _c(gu_bf16, np.uint16)
    dh = _c(dh_bf16, np.uint16)
    M, I2 = gu.shape
    I = I2 // 2
    assert dh.shape == (M, I)
    dgu = np.empty((M, 2 * I), dtype=np.uint16)
    alt = np.empty((M, 2 * I), dtype=np.uint16)
    n = _load().orc_silu_mul_bwd(_p(gu), _p(dh), M, I, _p(dgu), _p(alt))
    return dgu, alt, int(n)


def silu_mul_bwd_quant(gu_bf16, dh_bf16):
    """SiLU-mul backward, then the dual quantization of dGU: (q, s, qT, sT, dgu, alt)."""
    dgu, alt, _ = silu_mul_bwd(gu_bf16, dh_bf16)
    q, s = quantize_1x128(dgu)
    qT, sT = quantize_128x1(dgu) if dgu.shape[0] % 128 == 0 else (None, None)
    return q, s, qT, sT, dgu, alt


def rmsnorm_bwd(x_bf16, gamma_bf16, rstd, dy_bf16):
    """RMSNorm backward from the forward's rstd: (dx uint16 [M,K], mag float64 [M,K],
    dgamma float64 [K]); mag = |r*gamma*dy| + |r^3*x*S/K| per element."""
    x = _c(x_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    r = _c(rstd, np.float32)
    dy = _c(dy_bf16, np.uint16)
    M, K = x.shape
    dx = np.empty((M, K), dtype=np.uint16)
    mag = np.empty((M, K), dtype=np.float64)
    dgamma = np.empty(K, dtype=np.float64)
    _load().orc_rmsnorm_bwd(_p(x), _p(g), _p(r), _p(dy), M, K, _p(dx), _p(mag), _p(dgamma))
    return dx, mag, dgamma


def rmsnorm_quant(x_bf16, gamma_bf16, eps, rstd_in=None):
    """RMSNorm then the two quantizations of y: (q, s, qT, sT, rstd, y)."""
    y, r = rmsnorm(x_bf16, gamma_bf16, eps, rstd_in)
    q, s = quantize_1x128(y)
    qT, sT = quantize_128x1(y) if y.shape[0] % 128 == 0 else (None, None)
    return q, s, qT, sT, r, y


# ------------------------------------------------------------------ block-scaled GEMM

_MODES = ("fwd", "dgrad", "wgrad")


def _scale_strides(mode: str, R2: int, Kr: int):
    if mode == "fwd":       # B = W[N,K], scales [N/128, K/128]
        return 1, Kr // 128, 128
    if mode == "dgrad":     # B = W^T[K,N], scales of W: [N/128 (=kb), K/128 (=r2/128)]
        return R2 // 128, 1, 128
    if mode == "wgrad":     # B = X^T[K,M], scales [M/128 (=kb), K (=r2)]
        return R2, 1, 1
    raise ValueError(mode)


def gemm(A, sa, B, sb, mode: str):
    """Block-scaled C[R1,R2] = sum_kb sa(kb,r1) sb(kb,r2) (A_kb . B_kb) in binary64.

    A[R1,Kr], B[R2,Kr] uint8 codes (reduction contiguous); sa[Kr/128, R1];
    sb laid out as for ``mode`` (see ``_scale_strides``)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    R1, Kr = A.shape
    R2, Kr2 = B.shape
    assert Kr == Kr2 and Kr % 128 == 0
    sb_kb, sb_r, sb_rdiv = _scale_strides(mode, R2, Kr)
    y = np.empty((R1, R2), dtype=np.float64)
    _load().orc_gemm(_p(A), Kr, _p(sa), R1, _p(B), Kr, _p(sb), sb_kb, sb_r, sb_rdiv, R1, R2,
                     Kr, _p(y))
    return y


def gemm_sampled(A, sa, B, sb, mode: str, r1, r2):
    """The same as ``gemm`` but only at output positions (r1[i], r2[i])."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    R1, Kr = A.shape
    R2, _ = B.shape
    sb_kb, sb_r, sb_rdiv = _scale_strides(mode, R2, Kr)
    i1 = _c(r1, np.int64)
    i2 = _c(r2, np.int64)
    y = np.empty(i1.size, dtype=np.float64)
    _load().orc_gemm_sampled(_p(A), Kr, _p(sa), R1, _p(B), Kr, _p(sb), sb_kb, sb_r, sb_rdiv,
                             Kr, _p(i1), _p(i2), i1.size, _p(y))
    return y


# ------------------------------------------------------------------ NVFP4 (rollout format)

def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """E2M1 codes (low 4 bits) -> binary64 values."""
    lib = _load()
    table = np.array([lib.orc_e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return table[_c(codes, np.uint8) & 0xF]


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Finite binary32 values -> E2M1 codes (RNE, saturating at +-6), one per byte."""
    x = _c(v, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().orc_e2m1_encode_array(_p(x), _p(out), x.size)
    return out


def e2m1_encode_bits_range(first: int, count: int) -> np.ndarray:
    """E2M1 codes for every binary32 bit pattern first, first+1, ..., first+count-1."""
    out = np.empty(count, dtype=np.uint8)
    _load().orc_e2m1_encode_bits_range(first, count, _p(out))
    return out


def quantize_nvfp4(x_bf16: np.ndarray):
    """X[M,K] (BF16 bits) -> (q uint8 [M, K/2] packed E2M1, sf uint8 [M, K/16] E4M3 block
    scales, g float32 [M] per-row scales)."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 16 == 0
    q = np.empty((M, K // 2), dtype=np.uint8)
    sf = np.empty((M, K // 16), dtype=np.uint8)
    g = np.empty(M, dtype=np.float32)
    _load().orc_quantize_nvfp4(_p(x), M, K, K, _p(q), _p(sf), _p(g))
    return q, sf, g


def gemm_nvfp4(qx, sfx, gx, qw, sfw, gw):
    """y[M,N] = gx[m] gw[n] sum_k e2m1(x) sbx e2m1(w) sbw in binary64 (unrounded)."""
    qx, qw = _c(qx, np.uint8), _c(qw, np.uint8)
    sfx, sfw = _c(sfx, np.uint8), _c(sfw, np.uint8)
    gx, gw = _c(gx, np.float32), _c(gw, np.float32)
    M, K2 = qx.shape
    N, K2w = qw.shape
    assert K2 == K2w and sfx.shape == (M, K2 // 8) and sfw.shape == (N, K2 // 8)
    y = np.empty((M, N), dtype=np.float64)
    _load().orc_gemm_nvfp4(_p(qx), _p(sfx), _p(gx), M, _p(qw), _p(sfw), _p(gw), N, 2 * K2, _p(y))
    return y


def gemm_nvfp4_sampled(qx, sfx, gx, qw, sfw, gw, m, n):
    """The same as ``gemm_nvfp4`` at output positions (m[i], n[i]) only."""
    qx, qw = _c(qx, np.uint8), _c(qw, np.uint8)
    sfx, sfw = _c(sfx, np.uint8), _c(sfw, np.uint8)
    gx, gw = _c(gx, np.float32), _c(gw, np.float32)
    K = 2 * qx.shape[1]
    im, inn = _c(m, np.int64), _c(n, np.int64)
    y = np.empty(im.size, dtype=np.float64)
    _load().orc_gemm_nvfp4_sampled(_p(qx), _p(sfx), _p(gx), _p(qw), _p(sfw), _p(gw), K, _p(im), _p(inn),
                                   im.size, _p(y))
    return y
