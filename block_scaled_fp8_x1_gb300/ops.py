"""Torch-facing binding of libfp8rl: argument marshalling only.

Every function here hands raw device pointers, sizes and the current CUDA stream to the C
ABI (same names without the ``fp8rl_`` prefix); all arithmetic runs in the CUDA kernels.
PyTorch supplies the device memory (outputs are allocated with ``torch.empty``) and the
stream.  BF16 tensors travel as their bit patterns, E4M3 codes as ``torch.uint8`` (a
``torch.float8_e4m3fn`` view is available through ``as_e4m3``), scales as ``float32``.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional

import torch

from . import _abi
from ._abi import GemmOpts, check, lib


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _require(t: torch.Tensor, dtype: torch.dtype, name: str, device=None) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def _contig(t: torch.Tensor, name: str) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")


def _out(out: Optional[torch.Tensor], shape, device) -> torch.Tensor:
    """A caller-given output (bf16, on `device`, of `shape`, contiguous: the C calls write it
    with row stride shape[1]) or a new one."""
    if out is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    _require(out, torch.bfloat16, "out", device)
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out: expected shape {tuple(shape)}, got {tuple(out.shape)}")
    _contig(out, "out")
    return out


def as_e4m3(q: torch.Tensor) -> torch.Tensor:
    """View uint8 codes as torch.float8_e4m3fn (no copy)."""
    return q.view(torch.float8_e4m3fn)


# ------------------------------------------------------------------ status / diagnostics

def version() -> int:
    return lib().fp8rl_version()


def init(device: int = 0) -> None:
    check(lib().fp8rl_init(int(device)), "fp8rl_init")


def set_wait_timeout_ns(ns: int) -> None:
    lib().fp8rl_set_wait_timeout_ns(int(ns))


def check_status(device: Optional[torch.device] = None) -> int:
    """Wait for the current stream and return (and clear) the device status word."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    return int(lib().fp8rl_check_status(_stream(device)))


def debug_e4m3_encode(v: torch.Tensor) -> torch.Tensor:
    _require(v, torch.float32, "v")
    _contig(v, "v")
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    check(lib().fp8rl_debug_e4m3_encode(_ptr(v), _ptr(out), v.numel(), _stream(v.device)),
          "fp8rl_debug_e4m3_encode")
    return out


def debug_e2m1_encode(v: torch.Tensor) -> torch.Tensor:
    _require(v, torch.float32, "v")
    _contig(v, "v")
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    check(lib().fp8rl_debug_e2m1_encode(_ptr(v), _ptr(out), v.numel(), _stream(v.device)),
          "fp8rl_debug_e2m1_encode")
    return out


def debug_encode_check(amax_lo: int = 1, amax_hi: int = 0x7F80):
    """(mismatches, first_bad) of the division-free encode vs IEEE division over every BF16
    group maximum in [amax_lo, amax_hi) and every BF16 x with |x| <= amax."""
    dev = torch.device("cuda", torch.cuda.current_device())
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    first = torch.full((1,), -1, dtype=torch.int32, device=dev)
    check(lib().fp8rl_debug_encode_check(int(amax_lo), int(amax_hi), _ptr(cnt), _ptr(first),
                                         _stream(dev)), "fp8rl_debug_encode_check")
    torch.cuda.synchronize(dev)
    return int(cnt.item()), int(first.item()) & 0xFFFFFFFF


def debug_wait_timeout(timeout_ns: int, device: Optional[torch.device] = None) -> None:
    device = device or torch.device("cuda", torch.cuda.current_device())
    check(lib().fp8rl_debug_wait_timeout(int(timeout_ns), _stream(device)),
          "fp8rl_debug_wait_timeout")


# ------------------------------------------------------------------ quantizers

def quantize_1x128(x: torch.Tensor, dual: bool = False):
    """x bf16 [M,K] -> (q u8 [M,K], s f32 [K/128,M]) and, if dual, (qT [K,M], sT [M/128,K])."""
    _require(x, torch.bfloat16, "x")
    M, K = x.shape
    if x.stride(1) != 1:
        raise ValueError("x: rows must be contiguous")
    dev = x.device
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    qT = sT = None
    if dual:
        qT = torch.empty((K, M), dtype=torch.uint8, device=dev)
        sT = torch.empty((M // 128, K), dtype=torch.float32, device=dev)
    check(lib().fp8rl_quantize_1x128(_ptr(x), M, K, x.stride(0), _ptr(q), _ptr(s), _ptr(qT),
                                     _ptr(sT), _stream(dev)), "fp8rl_quantize_1x128")
    return (q, s, qT, sT) if dual else (q, s)


def quantize_128x1(x: torch.Tensor):
    """x bf16 [M,K] -> (qT u8 [K,M], sT f32 [M/128,K])."""
    _require(x, torch.bfloat16, "x")
    M, K = x.shape
    if x.stride(1) != 1:
        raise ValueError("x: rows must be contiguous")
    dev = x.device
    qT = torch.empty((K, M), dtype=torch.uint8, device=dev)
    sT = torch.empty((M // 128, K), dtype=torch.float32, device=dev)
    check(lib().fp8rl_quantize_128x1(_ptr(x), M, K, x.stride(0), _ptr(qT), _ptr(sT),
                                     _stream(dev)), "fp8rl_quantize_128x1")
    return qT, sT


def requantize_128x1(q: torch.Tensor, s: torch.Tensor):
    """From a saved 1x128 quantization (q u8 [M,K], s f32 [K/128,M]): the 128x1 WGrad operand
    of the dequantized BF16 activation, transposed: (qT u8 [K,M], sT f32 [M/128,K])."""
    _require(q, torch.uint8, "q")
    _require(s, torch.float32, "s", q.device)
    _contig(q, "q")
    _contig(s, "s")
    M, K = q.shape
    dev = q.device
    qT = torch.empty((K, M), dtype=torch.uint8, device=dev)
    sT = torch.empty((M // 128, K), dtype=torch.float32, device=dev)
    check(lib().fp8rl_requantize_128x1(_ptr(q), _ptr(s), M, K, _ptr(qT), _ptr(sT), _stream(dev)),
          "fp8rl_requantize_128x1")
    return qT, sT


def quantize_128x128(w: torch.Tensor, transpose: bool = True):
    """w bf16 [N,K] -> (q u8 [N,K], s f32 [N/128,K/128], qT u8 [K,N] or None)."""
    _require(w, torch.bfloat16, "w")
    N, K = w.shape
    if w.stride(1) != 1:
        raise ValueError("w: rows must be contiguous")
    dev = w.device
    q = torch.empty((N, K), dtype=torch.uint8, device=dev)
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    qT = torch.empty((K, N), dtype=torch.uint8, device=dev) if transpose else None
    check(lib().fp8rl_quantize_128x128(_ptr(w), N, K, w.stride(0), _ptr(q), _ptr(s), _ptr(qT),
                                       _stream(dev)), "fp8rl_quantize_128x128")
    return q, s, qT


def rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float, dual: bool = True):
    """Fused RMSNorm -> quantize: (q, s, qT, sT, rstd); qT/sT are None unless dual."""
    _require(x, torch.bfloat16, "x")
    _require(gamma, torch.bfloat16, "gamma", x.device)
    _contig(x, "x")
    _contig(gamma, "gamma")
    M, K = x.shape
    dev = x.device
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    rstd = torch.empty((M,), dtype=torch.float32, device=dev)
    qT = sT = None
    if dual:
        qT = torch.empty((K, M), dtype=torch.uint8, device=dev)
        sT = torch.empty((M // 128, K), dtype=torch.float32, device=dev)
    check(lib().fp8rl_rmsnorm_quant(_ptr(x), _ptr(gamma), ctypes.c_float(eps), M, K, _ptr(q),
                                    _ptr(s), _ptr(qT), _ptr(sT), _ptr(rstd), _stream(dev)),
          "fp8rl_rmsnorm_quant")
    return q, s, qT, sT, rstd


def silu_mul_quant(gu: torch.Tensor, dual: bool = True):
    """gu bf16 [M, 2I] -> (q [M,I], s [I/128,M], qT [I,M] or None, sT [M/128,I] or None)."""
    _require(gu, torch.bfloat16, "gu")
    _contig(gu, "gu")
    M, I2 = gu.shape
    I = I2 // 2
    dev = gu.device
    q = torch.empty((M, I), dtype=torch.uint8, device=dev)
    s = torch.empty((I // 128, M), dtype=torch.float32, device=dev)
    qT = sT = None
    if dual:
        qT = torch.empty((I, M), dtype=torch.uint8, device=dev)
        sT = torch.empty((M // 128, I), dtype=torch.float32, device=dev)
    check(lib().fp8rl_silu_mul_quant(_ptr(gu), M, I, _ptr(q), _ptr(s), _ptr(qT), _ptr(sT),
                                     _stream(dev)), "fp8rl_silu_mul_quant")
    return q, s, qT, sT


# ------------------------------------------------------------------ backward steps

def silu_mul_bwd_quant(gu: torch.Tensor, dh: torch.Tensor, dual: bool = True):
    """Gradient of the gate_up output from the forward's gu bf16 [M, 2I] and dh bf16 [M, I],
    quantized: (q [M,2I], s [2I/128,M], qT [2I,M] or None, sT [M/128,2I] or None)."""
    _require(gu, torch.bfloat16, "gu")
    _require(dh, torch.bfloat16, "dh", gu.device)
    _contig(gu, "gu")
    _contig(dh, "dh")
    M, I2 = gu.shape
    if dh.shape != (M, I2 // 2):
        raise ValueError(f"dh: expected {(M, I2 // 2)}, got {tuple(dh.shape)}")
    dev = gu.device
    q = torch.empty((M, I2), dtype=torch.uint8, device=dev)
    s = torch.empty((I2 // 128, M), dtype=torch.float32, device=dev)
    qT = sT = None
    if dual:
        qT = torch.empty((I2, M), dtype=torch.uint8, device=dev)
        sT = torch.empty((M // 128, I2), dtype=torch.float32, device=dev)
    check(lib().fp8rl_silu_mul_bwd_quant(_ptr(gu), _ptr(dh), M, I2 // 2, _ptr(q), _ptr(s), _ptr(qT),
                                         _ptr(sT), _stream(dev)), "fp8rl_silu_mul_bwd_quant")
    return q, s, qT, sT


def rmsnorm_bwd(x: torch.Tensor, gamma: torch.Tensor, rstd: torch.Tensor, dy: torch.Tensor,
                with_dgamma: bool = True):
    """RMSNorm backward from the forward's rstd: (dx bf16 [M,K], dgamma f32 [K] or None)."""
    _require(x, torch.bfloat16, "x")
    _require(gamma, torch.bfloat16, "gamma", x.device)
    _require(rstd, torch.float32, "rstd", x.device)
    _require(dy, torch.bfloat16, "dy", x.device)
    for t, n in ((x, "x"), (gamma, "gamma"), (rstd, "rstd"), (dy, "dy")):
        _contig(t, n)
    M, K = x.shape
    dev = x.device
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dgamma = ws = None
    if with_dgamma:
        dgamma = torch.empty((K,), dtype=torch.float32, device=dev)
        ws = workspace(int(lib().fp8rl_rmsnorm_bwd_workspace_bytes(M, K)), dev)
    check(lib().fp8rl_rmsnorm_bwd(_ptr(x), _ptr(gamma), _ptr(rstd), _ptr(dy), M, K, _ptr(dx),
                                  _ptr(dgamma), _ptr(ws), ws.numel() if ws is not None else 0,
                                  _stream(dev)), "fp8rl_rmsnorm_bwd")
    return dx, dgamma


# ------------------------------------------------------------------ GEMMs

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def gemm_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return int(lib().fp8rl_gemm_workspace_bytes(int(op), M, N, K))


def workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """A byte buffer of at least nbytes, cached per device.

    It holds the decode form's split-K partial sums, which every call writes before it
    reads them, so one buffer serves every call issued in stream order on that device."""
    key = (device.type, device.index)
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = buf
        return buf


def _check_gemm_inputs(qa, sa, qb, sb):
    _require(qa, torch.uint8, "codes A")
    _require(qb, torch.uint8, "codes B", qa.device)
    _require(sa, torch.float32, "scales A", qa.device)
    _require(sb, torch.float32, "scales B", qa.device)
    for t, n in ((qa, "codes A"), (qb, "codes B"), (sa, "scales A"), (sb, "scales B")):
        _contig(t, n)


def gemm_fwd(qx, sx, qw, sw, out=None, variant: int = _abi.FP8RL_VARIANT_AUTO, splits: int = 0,
             grid: int = 0, ws: Optional[torch.Tensor] = None, tile_n: int = 0, epi_warps: int = 0):
    """Y = X W^T: qx [M,K], sx [K/128,M], qw [N,K], sw [N/128,K/128] -> y bf16 [M,N]."""
    _check_gemm_inputs(qx, sx, qw, sw)
    M, K = qx.shape
    N = qw.shape[0]
    dev = qx.device
    y = _out(out, (M, N), dev)
    opts = GemmOpts(int(variant), int(splits), int(grid), int(tile_n), int(epi_warps))
    wsb = ws
    need = int(lib().fp8rl_gemm_workspace_bytes_ex(_abi.FP8RL_OP_FWD, M, N, K, ctypes.byref(opts)))
    if need > 0 and wsb is None:
        wsb = workspace(need, dev)
    check(lib().fp8rl_gemm_fwd_ex(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(y), M, N, K,
                                  _ptr(wsb), wsb.numel() if wsb is not None else 0,
                                  ctypes.byref(opts), _stream(dev)), "fp8rl_gemm_fwd_ex")
    return y


def gemm_dgrad(qdy, sdy, qwT, sw, out=None, variant: int = _abi.FP8RL_VARIANT_AUTO,
               grid: int = 0, epi_warps: int = 0, tile_n: int = 0):
    """dX = dY W: qdy [M,N], sdy [N/128,M], qwT [K,N], sw [N/128,K/128] -> dx bf16 [M,K]."""
    _check_gemm_inputs(qdy, sdy, qwT, sw)
    M, N = qdy.shape
    K = qwT.shape[0]
    dev = qdy.device
    dx = _out(out, (M, K), dev)
    opts = GemmOpts(int(variant), 0, int(grid), int(tile_n), int(epi_warps))
    check(lib().fp8rl_gemm_dgrad_ex(_ptr(qdy), _ptr(sdy), _ptr(qwT), _ptr(sw), _ptr(dx), M, N, K,
                                    None, 0, ctypes.byref(opts), _stream(dev)), "fp8rl_gemm_dgrad_ex")
    return dx


def gemm_wgrad(qdyT, sdyT, qxT, sxT, out=None, variant: int = _abi.FP8RL_VARIANT_AUTO,
               grid: int = 0, epi_warps: int = 0, tile_n: int = 0):
    """dW = dY^T X: qdyT [N,M], sdyT [M/128,N], qxT [K,M], sxT [M/128,K] -> dw bf16 [N,K]."""
    _check_gemm_inputs(qdyT, sdyT, qxT, sxT)
    N, M = qdyT.shape
    K = qxT.shape[0]
    dev = qdyT.device
    dw = _out(out, (N, K), dev)
    opts = GemmOpts(int(variant), 0, int(grid), int(tile_n), int(epi_warps))
    check(lib().fp8rl_gemm_wgrad_ex(_ptr(qdyT), _ptr(sdyT), _ptr(qxT), _ptr(sxT), _ptr(dw), M, N,
                                    K, None, 0, ctypes.byref(opts), _stream(dev)), "fp8rl_gemm_wgrad_ex")
    return dw


def linear_fwd(x: torch.Tensor, qw, sw, out=None):
    """One linear layer from the BF16 activation: x bf16 [M,K] is quantized 1x128 (returned
    as qx u8 [M,K], sx f32 [K/128,M]) and y = X W^T bf16 [M,N] computed from it; for
    M <= 256 the GEMM overlaps the quantizer.  Returns (y, qx, sx)."""
    _require(x, torch.bfloat16, "x")
    _require(qw, torch.uint8, "codes W", x.device)
    _require(sw, torch.float32, "scales W", x.device)
    _contig(qw, "codes W")
    _contig(sw, "scales W")
    if x.stride(1) != 1:
        raise ValueError("x: rows must be contiguous")
    M, K = x.shape
    N = qw.shape[0]
    dev = x.device
    qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    y = _out(out, (M, N), dev)
    need = gemm_workspace_bytes(_abi.FP8RL_OP_FWD, M, N, K)
    wsb = workspace(need, dev) if need > 0 else None
    check(lib().fp8rl_linear_fwd(_ptr(x), M, K, x.stride(0), _ptr(qw), _ptr(sw), N, _ptr(qx),
                                 _ptr(sx), _ptr(y), _ptr(wsb), wsb.numel() if wsb is not None else 0,
                                 _stream(dev)), "fp8rl_linear_fwd")
    return y, qx, sx


# ------------------------------------------------------------------ NVFP4 rollout path

def nvfp4_scale_bytes(R: int, K: int) -> int:
    return int(lib().fp8rl_nvfp4_scale_bytes(R, K))


def _nvfp4_buffers(R: int, K: int, dev):
    q = torch.empty((R, K // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty(nvfp4_scale_bytes(R, K), dtype=torch.uint8, device=dev)
    g = torch.empty(R, dtype=torch.float32, device=dev)
    return q, sf, g


def quantize_nvfp4(x: torch.Tensor):
    """NVFP4 quantization of the rows of x bf16 [R,K] (K % 256 == 0): (q u8 [R, K/2] packed
    E2M1, sf u8 block scales in the tensor core's atom layout, g f32 [R])."""
    _require(x, torch.bfloat16, "x")
    if x.stride(1) != 1:
        raise ValueError("x: rows must be contiguous")
    R, K = x.shape
    q, sf, g = _nvfp4_buffers(R, K, x.device)
    check(lib().fp8rl_quantize_nvfp4(_ptr(x), R, K, x.stride(0), _ptr(q), _ptr(sf), _ptr(g),
                                     _stream(x.device)), "fp8rl_quantize_nvfp4")
    return q, sf, g


def gemm_nvfp4(qx, sfx, gx, qw, sfw, gw, splits: int = 0, out=None):
    """y bf16 [M,N] from NVFP4 operands of X [M,K] and W [N,K] (decode shapes, M <= 256)."""
    dev = qx.device
    for t, n, dt in ((qx, "qx", torch.uint8), (sfx, "sfx", torch.uint8), (gx, "gx", torch.float32),
                     (qw, "qw", torch.uint8), (sfw, "sfw", torch.uint8), (gw, "gw", torch.float32)):
        _require(t, dt, n, dev)
        _contig(t, n)
    M, K2 = qx.shape
    N = qw.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    _require(y, torch.bfloat16, "out", dev)
    if y.shape != (M, N) or y.stride(1) != 1:
        raise ValueError("out: expected a [M, N] bf16 view with contiguous rows")
    check(lib().fp8rl_gemm_nvfp4(_ptr(qx), _ptr(sfx), _ptr(gx), _ptr(qw), _ptr(sfw), _ptr(gw), _ptr(y),
                                 M, N, 2 * K2, y.stride(0), int(splits), _stream(dev)), "fp8rl_gemm_nvfp4")
    return y


def linear_nvfp4(x: torch.Tensor, qw, sfw, gw, out=None):
    """One NVFP4 linear layer from the BF16 activation x [M,K]: the activation's NVFP4
    operands and y = X W^T bf16 [M,N].  Returns (y, qx, sfx, gx)."""
    _require(x, torch.bfloat16, "x")
    if x.stride(1) != 1:
        raise ValueError("x: rows must be contiguous")
    M, K = x.shape
    N = qw.shape[0]
    dev = x.device
    qx, sfx, gx = _nvfp4_buffers(M, K, dev)
    y = _out(out, (M, N), dev)
    check(lib().fp8rl_linear_nvfp4(_ptr(x), M, K, x.stride(0), _ptr(qw), _ptr(sfw), _ptr(gw), N, _ptr(qx),
                                   _ptr(sfx), _ptr(gx), _ptr(y), _stream(dev)), "fp8rl_linear_nvfp4")
    return y, qx, sfx, gx
