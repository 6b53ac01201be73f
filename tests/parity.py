"""Comparison helpers shared by the GPU parity tests (test infrastructure).

The tolerance of a GEMM output is the one the build targets for the block-scaled FP8
linear layer: elementwise |y - y_ref| <= 2^-7 |y_ref| + 1e-3 * rms(y_ref), with y_ref the
oracle's unrounded binary64 result.  Quantized codes and scales must be bit-exact.
"""
from __future__ import annotations

import itertools

import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def assert_same_bits_f32(a: np.ndarray, b: np.ndarray, what: str) -> None:
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    bad = a.view(np.uint32) != b.view(np.uint32)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {a.size} differ, first at {np.argwhere(bad)[0]}"


def assert_same_u8(a: np.ndarray, b: np.ndarray, what: str) -> None:
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    bad = a != b
    assert not bad.any(), f"{what}: {int(bad.sum())} of {a.size} codes differ, first at {np.argwhere(bad)[0]}"


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_tolerance_check(y_bits: np.ndarray, y_ref: np.ndarray, what: str,
                         rms: float | None = None) -> dict:
    """Elementwise bound; returns statistics (max normalised error, share equal to the
    round-to-nearest BF16 of y_ref)."""
    y = bf16_bits_to_f64(y_bits)
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    bound = 2.0 ** -7 * np.abs(y_ref) + 1e-3 * rms
    err = np.abs(y - y_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {y.size} outside the bound; worst "
                           f"{float(np.max(err - bound)):.3e} at {np.argwhere(bad)[0]}")
    rne = torch.from_numpy(y_ref).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return {"max_err_over_bound": float(np.max(err / np.maximum(bound, 1e-300))) if y.size else 0.0,
            "rne_equal_share": float(np.mean(rne == y_bits)) if y.size else 1.0}


def silu_group_matches(oracle, gpu_codes: np.ndarray, gpu_scale: np.float32, h: np.ndarray,
                       alt: np.ndarray, max_flagged: int = 12) -> bool:
    """A group of SiLU-mul outputs matches if the GPU's codes and scale equal the oracle's
    quantization of some choice between h and alt at the flagged elements (where a binary32
    evaluation may round to either BF16 neighbour)."""
    flagged = np.nonzero(h != alt)[0]
    if len(flagged) > max_flagged:
        flagged = flagged[:max_flagged]
    for choice in itertools.product((0, 1), repeat=len(flagged)):
        v = h.copy()
        for sel, idx in zip(choice, flagged):
            if sel:
                v[idx] = alt[idx]
        q, s = oracle.quant_group(oracle.bf16_to_f32(v))
        if np.float32(s).view(np.uint32) == np.float32(gpu_scale).view(np.uint32) and np.array_equal(q, gpu_codes):
            return True
    return False
