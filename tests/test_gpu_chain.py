"""One transformer layer's FP8 linear chain, rollout form against training form.

"Technical summary: Jet-RL", section "Core architecture": the inference (rollout) graph is
a sub-graph of the training forward graph, with the same quantization granularity and
precision.  The chain here is the layer's linear path:

    rmsnorm_quant(x) -> qkv -> [attention: out of scope; a seeded stand-in for its output]
    -> quantize -> o -> residual x + o -> rmsnorm_quant -> gate_up -> silu_mul_quant -> down

run once over a training batch (tiled GEMMs) and once over a subset of its rows as rollout
would (decode-shaped GEMMs).  Every quantizer is row-wise, and the decode form without a
split of the reduction adds the same per-K-block products in the same order as the tiled
form, so the rollout rows must reproduce the training rows' FP8 codes, scales and BF16
outputs bit for bit at every stage.  With the automatic decode choice (which may split the
reduction inside a cluster) the outputs stay within the GEMM bound of the oracle and the
codes are the oracle's quantization of their own inputs.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth
from parity import assert_same_bits_f32, assert_same_u8, bits16, f32, gemm_tolerance_check, u8

pytestmark = pytest.mark.gpu

H, NQKV, I = 1024, 1536, 2816       # hidden, qkv width, intermediate (all multiples of 128)


def layer_weights(fp8lib):
    w = {}
    for i, (name, (N, K)) in enumerate({"qkv": (NQKV, H), "o": (H, H), "gate_up": (2 * I, H),
                                        "down": (H, I)}.items()):
        wt = synth.normal_bf16((N, K), 0.02, 500 + i, "cuda")
        w[name] = fp8lib.quantize_128x128(wt, transpose=False)[:2]
    return w


def chain(fp8lib, w, x, attn, gamma, variant, splits=0):
    """The layer's linear path; returns every FP8 tensor and BF16 output in order."""
    out = {}

    def gemm(name, q, s):
        return fp8lib.gemm_fwd(q, s, w[name][0], w[name][1], variant=variant, splits=splits)

    q, s, _, _, _ = fp8lib.rmsnorm_quant(x, gamma, 1e-5, dual=False)
    out["x_q"], out["x_s"] = q, s
    out["qkv"] = gemm("qkv", q, s)
    q, s = fp8lib.quantize_1x128(attn)
    out["attn_q"], out["attn_s"] = q, s
    out["o"] = gemm("o", q, s)
    h = (x.float() + out["o"].float()).to(torch.bfloat16)        # residual (BF16)
    q, s, _, _, _ = fp8lib.rmsnorm_quant(h, gamma, 1e-5, dual=False)
    out["h_q"], out["h_s"] = q, s
    out["gate_up"] = gemm("gate_up", q, s)
    q, s, _, _ = fp8lib.silu_mul_quant(out["gate_up"], dual=False)
    out["act_q"], out["act_s"] = q, s
    out["y"] = gemm("down", q, s)
    return out


def rows_of(name, t, rows):
    """Rows of a chain tensor: codes and outputs are [M, *], scales [*, M]."""
    return t[:, rows] if name.endswith("_s") else t[rows]


@pytest.mark.parametrize("rows", [slice(64, 128), slice(0, 200), slice(300, 301)])
def test_rollout_rows_reproduce_training_bytes(fp8lib, oracle, rows):
    M = 512
    x = synth.normal_bf16((M, H), 1.0, 71, "cuda", outlier_channels=2, outlier_scale=30.0)
    attn = synth.normal_bf16((M, H), 1.0, 72, "cuda")
    gamma = synth.normal_bf16((H,), 0.1, 73, "cuda").float().add_(1.0).to(torch.bfloat16)
    w = layer_weights(fp8lib)
    train = chain(fp8lib, w, x, attn, gamma, _abi.FP8RL_VARIANT_TILED)
    xs, ats = x[rows].contiguous(), attn[rows].contiguous()
    roll = chain(fp8lib, w, xs, ats, gamma, _abi.FP8RL_VARIANT_DECODE, splits=1)
    for name, t in train.items():
        a = rows_of(name, t, rows).contiguous()
        b = roll[name]
        assert a.dtype == b.dtype and a.shape == b.shape, name
        if a.dtype == torch.float32:
            assert_same_bits_f32(f32(b), f32(a), f"rollout {name}")
        elif a.dtype == torch.uint8:
            assert_same_u8(u8(b), u8(a), f"rollout {name}")
        else:
            assert np.array_equal(bits16(b), bits16(a)), f"rollout {name}: BF16 outputs differ"
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_rollout_chain_with_automatic_decode_forms(fp8lib, oracle):
    M = 96
    x = synth.normal_bf16((M, H), 1.0, 81, "cuda", outlier_channels=2, outlier_scale=30.0)
    attn = synth.normal_bf16((M, H), 1.0, 82, "cuda")
    gamma = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    w = layer_weights(fp8lib)
    roll = chain(fp8lib, w, x, attn, gamma, _abi.FP8RL_VARIANT_AUTO)
    # each GEMM output against the oracle on that stage's own codes
    for out, (qn, sn), wn in (("qkv", ("x_q", "x_s"), "qkv"), ("o", ("attn_q", "attn_s"), "o"),
                              ("gate_up", ("h_q", "h_s"), "gate_up"), ("y", ("act_q", "act_s"), "down")):
        ref = oracle.gemm(u8(roll[qn]), f32(roll[sn]), u8(w[wn][0]), f32(w[wn][1]), "fwd")
        gemm_tolerance_check(bits16(roll[out]), ref, f"rollout {out}")
    # the quantized activations are the oracle's quantization of their inputs
    qa, sa = oracle.quantize_1x128(bits16(attn))
    assert_same_u8(u8(roll["attn_q"]), qa, "attention output codes")
    assert_same_bits_f32(f32(roll["attn_s"]), sa, "attention output scales")
