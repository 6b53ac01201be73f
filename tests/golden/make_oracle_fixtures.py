"""Writes tests/golden/oracle_small.txt and oracle_nvfp4_small.txt: the oracle's outputs on
tiny closed-form inputs.

Run from the repository root:  python tests/golden/make_oracle_fixtures.py
Calls only the CPU oracle (oracle/).  The pages of the scheme ("Technical summary:
Jet-RL") print no worked example, so this fixture is a regression record of the pinned
oracle, not an independent reference: a later change to the oracle's arithmetic that
alters these bytes must name the passage, or the reading of it, that justifies it.

Input (closed form, no random numbers):
  x[r, c] = bf16( (c - 100) * 0.0371 * (r + 1) ),  r < 4, c < 256    (activations)
  w[n, c] = bf16( ((7 * n + 3 * c) % 23 - 11) * 0.0023 ),  n < 128  (one weight block row)
Records: 1x128 codes/scales of x, the SHA-256 of w's 128x128 codes, w's scales, and
y = X W^T (binary64).  The NVFP4 file (the rollout format of the QeRL page) records the
NVFP4 codes, block scales and row scales of the same x and w and their product.
"""
import hashlib
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    return oracle.f64_to_bf16(np.asarray(a, dtype=np.float32).astype(np.float64))


def inputs():
    r = np.arange(4)[:, None]
    c = np.arange(256)[None, :]
    x = (c - 100) * 0.0371 * (r + 1)
    n = np.arange(128)[:, None]
    w = (((7 * n + 3 * c) % 23) - 11) * 0.0023
    return f32_to_bf16_bits(x), f32_to_bf16_bits(w)


def compute():
    xb, wb = inputs()
    qx, sx = oracle.quantize_1x128(xb)
    qw, sw, _ = oracle.quantize_128x128(wb)
    y = oracle.gemm(qx, sx, qw, sw, "fwd")
    return qx, sx, qw, sw, y


def render() -> str:
    qx, sx, qw, sw, y = compute()
    lines = ["# oracle regression fixture, written by tests/golden/make_oracle_fixtures.py"]
    lines.append("qx " + bytes(qx.ravel()).hex())
    lines.append("sx " + " ".join(float(v).hex() for v in sx.ravel()))
    lines.append("qw_sha256 " + hashlib.sha256(bytes(qw.ravel())).hexdigest())
    lines.append("sw " + " ".join(float(v).hex() for v in sw.ravel()))
    lines.append("y " + " ".join(float(v).hex() for v in y.ravel()))
    return "\n".join(lines) + "\n"


def render_nvfp4() -> str:
    xb, wb = inputs()
    qx, sx, gx = oracle.quantize_nvfp4(xb)
    qw, sw, gw = oracle.quantize_nvfp4(wb)
    y = oracle.gemm_nvfp4(qx, sx, gx, qw, sw, gw)
    lines = ["# oracle NVFP4 regression fixture, written by tests/golden/make_oracle_fixtures.py"]
    lines.append("qx " + bytes(qx.ravel()).hex())
    lines.append("sfx " + bytes(sx.ravel()).hex())
    lines.append("gx " + " ".join(float(v).hex() for v in gx.ravel()))
    lines.append("qw_sha256 " + hashlib.sha256(bytes(qw.ravel())).hexdigest())
    lines.append("sfw " + bytes(sw.ravel()).hex())
    lines.append("gw " + " ".join(float(v).hex() for v in gw.ravel()))
    lines.append("y " + " ".join(float(v).hex() for v in y.ravel()))
    return "\n".join(lines) + "\n"


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.txt"), "w") as f:
        f.write(render())
    with open(os.path.join(HERE, "oracle_nvfp4_small.txt"), "w") as f:
        f.write(render_nvfp4())
    print("wrote oracle_small.txt, oracle_nvfp4_small.txt")
