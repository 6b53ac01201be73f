"""block_scaled_fp8_x1_gb300 -- unified-precision FP8 linear layer for GB300 (sm_103a).

The compute lives in ``libfp8rl.so`` (CUDA kernels behind the C ABI of
``include/fp8rl.h``); ``ops`` marshals torch tensors into those calls.  The library is
loaded on the first call and its absence is an error: there is no CPU fallback.
"""
from . import ops, synth  # noqa: F401

__all__ = ["ops", "synth", "build_library"]


def build_library(force: bool = False) -> str:
    from .build import build
    return build(force=force)
