"""Benchmark of the unified-precision FP8 linear layer on one GB300 (or N replicas).

One step = one pass of the whole hot path over a Qwen2.5-32B-shaped transformer layer at
16384 tokens (hidden 5120; qkv 7168x5120, o 5120x5120, gate_up 55296x5120, down
5120x27648), forward, DGrad and WGrad of all four linears with their quantizers
("Technical summary: Jet-RL": rollout and training forward share one quantization flow;
master weights stay BF16 and are re-quantized each step; DGrad and WGrad run in FP8):

  weight refresh   quantize_128x128(W) for qkv, o, gate_up, down  (+ W^T copies)
  forward          rmsnorm_quant(X_attn) -> gemm_fwd(qkv)
                   quantize_1x128 dual(attention output) -> gemm_fwd(o)
                   rmsnorm_quant(X_mlp) -> gemm_fwd(gate_up) -> silu_mul_quant -> gemm_fwd(down)
  backward         for each linear: dual-quantized dY -> gemm_dgrad -> gemm_wgrad, where dY
                   is quantize_1x128 dual(dY) for qkv, o and down, and for gate_up
                   silu_mul_bwd_quant(gate_up output, dH = the DGrad of down)

value = GEMM FLOPs of the step / device time of the step (TFLOP/s), inputs resident in HBM
and larger than L2.  e2e = the same with the step's batch tensors (the three input
activations and the output gradients of qkv, o and down, 1.1 GB) copied from pinned host
memory and its results (the layer output and the four weight gradients, 1.1 GB) copied
back inside the timed region; the BF16 weights are model state on the device, re-quantized by the step.  Per-kernel CUDA-event times give the
quantizers' GB/s and the roofline of the dominant kernel.  Two more workloads are reported
beside it: the Llama-3.1-8B MLP training step at 8192 tokens, and the rollout decode
linears of Qwen2.5-7B at 64, 128 and 256 tokens (CUDA-graph replays over weight copies
larger than L2).

`--impl reference` times the CPU oracle (test infrastructure, unchanged) on the host cores
on a bounded sample of the same step and reports the same metric.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 block-scaled GEMM TFLOP/s & % FP8 peak; quantize GB/s vs HBM peak"
FP8_PER_BF16 = 2.0       # nominal dense FP8 / BF16 tensor throughput ratio on GB300
FP8_NOMINAL_TFLOPS = 4500.0

# Qwen2.5-32B-shaped layer at 16384 tokens (the headline step)
M32, H32 = 16384, 5120
LIN32 = {"qkv": (7168, 5120), "o": (5120, 5120), "gate_up": (55296, 5120), "down": (5120, 27648)}
WORKLOAD = ("Qwen2.5-32B layer at 16384 tokens: qkv 7168x5120, o 5120x5120, gate_up "
            "55296x5120, down 5120x27648; fwd + DGrad + WGrad of all four with their "
            "quantizers and the weight refresh; dY of gate_up from dH through the SiLU-mul "
            "backward")
# Llama-3.1-8B MLP at 8192 tokens (reported beside it)
M_TOK, HID, INTER = 8192, 4096, 14336
# Qwen2.5-7B decode linears (reported beside it)
DEC7B = {"qkv": (4608, 3584), "o": (3584, 3584), "gate_up": (37888, 3584), "down": (3584, 18944)}
DEC_M = (64, 128, 256)


def dual_bytes(E):
    """BF16 in, 1x128 and 128x1 codes and scales out."""
    return 2 * E + 2 * E + 2 * 4 * E / 128


def wq_bytes(E):
    """BF16 weight in, codes + W^T copy + block scales out."""
    return 2 * E + E + E + 4 * E / 16384


def silu_bytes(M, I):
    return 2 * 2 * M * I + M * I + M * I + 2 * 4 * M * I / 128


def silu_bwd_bytes(M, I):
    """gate_up output and dH in, the dual codes and scales of [dg | du] out."""
    return 2 * 2 * M * I + 2 * M * I + 2 * M * I + 2 * M * I + 2 * 4 * 2 * M * I / 128


def rms_bytes(M, K):
    return dual_bytes(M * K) + 2 * K + 4 * M


def layer32_work():
    """(GEMM FLOPs per launch name, algorithmic HBM bytes per quantizer launch name)."""
    f, b = {}, {}
    M = M32
    for name, (N, K) in LIN32.items():
        fl = 2.0 * M * N * K
        f[f"fwd_{name}"] = f[f"dgrad_{name}"] = f[f"wgrad_{name}"] = fl
        b[f"wq_{name}"] = wq_bytes(N * K)
        if name != "gate_up":
            b[f"dq_dy_{name}"] = dual_bytes(M * N)
    b["silu_mul_bwd_quant"] = silu_bwd_bytes(M, LIN32["down"][1])
    b["rmsnorm_quant_attn"] = rms_bytes(M, H32)
    b["dq_attn_out"] = dual_bytes(M * H32)
    b["rmsnorm_quant_mlp"] = rms_bytes(M, H32)
    b["silu_mul_quant"] = silu_bytes(M, LIN32["down"][1])
    return f, b


def mlp8_work():
    f, b = {}, {}
    f["fwd_gate_up"] = f["dgrad_gate_up"] = f["wgrad_gate_up"] = 2.0 * M_TOK * 2 * INTER * HID
    f["fwd_down"] = f["dgrad_down"] = f["wgrad_down"] = 2.0 * M_TOK * HID * INTER
    b["wq_gate_up"] = wq_bytes(2 * INTER * HID)
    b["wq_down"] = wq_bytes(HID * INTER)
    b["rmsnorm_quant"] = rms_bytes(M_TOK, HID)
    b["silu_mul_quant"] = silu_bytes(M_TOK, INTER)
    b["dq_dy_down"] = dual_bytes(M_TOK * HID)
    b["silu_mul_bwd_quant"] = silu_bwd_bytes(M_TOK, INTER)
    return f, b


def decode_work(M, N, K):
    """(FLOPs, algorithmic HBM bytes) of one decode-shaped linear: the FP8 weight stream and
    its block scales, the BF16 activations in, the BF16 output."""
    return 2.0 * M * N * K, N * K + 4 * (N // 128) * (K // 128) + 2 * M * K + 2 * M * N


def decode_work_nvfp4(M, N, K):
    """(FLOPs, algorithmic HBM bytes) of one NVFP4 decode linear: the packed E2M1 weights,
    their E4M3 block scales (one per 16) and row scales, the BF16 activations in, the BF16
    output."""
    return 2.0 * M * N * K, N * K // 2 + N * K // 16 + 4 * N + 2 * M * K + 2 * M * N


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples every 20 ms, kept only when their timestamp falls
    inside the window passed to stop()."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples (the JSON line keeps their summary); BENCH_CLOCKS_DIR keeps them elsewhere
        self.path = os.path.join(os.environ.get("BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        """Start sampling and return once the first sample is written (at most 5 s)."""
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t_end = time.time() + 5.0
        while time.time() < t_end and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self, window):
        """Stop sampling; summarise the samples taken between window[0] and window[1]
        (time.time() values)."""
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(p[2]), float(p[3]), float(p[4]), p[6], p[7], p[8], p[9]))
            except ValueError:
                continue
        inside = [r for r in rows if window[0] <= r[0] <= window[1]]
        if not inside:
            return None
        reasons = set()
        for r in inside:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), r[4:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": sorted(reasons),
                "power_w_median": statistics.median(r[3] for r in inside),
                "samples": len(inside), "window_ms": round(1e3 * (window[1] - window[0]), 1)}


# ----------------------------------------------------------------------------- peaks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------- GPU arm

class _Marks:
    """Optional CUDA events after each launch (for the per-kernel split)."""

    def __init__(self, torch, marks):
        self.torch, self.marks = torch, marks

    def __call__(self, name):
        if self.marks is not None:
            e = self.torch.cuda.Event(enable_timing=True)
            e.record()
            self.marks.append((name, e))


class Layer32Step:
    """Qwen2.5-32B-shaped layer at 16384 tokens: all buffers resident on the device and the
    launches of one step in order."""

    # 4 weight, 2x2 RMSNorm, 1 dual, 4 fwd, 1 SiLU-mul, 4x3 backward (gate_up's gradient
    # quantizer being the SiLU-mul backward)
    LAUNCHES_PER_STEP = 26

    def __init__(self, dev):
        import torch
        from block_scaled_fp8_x1_gb300 import _abi, ops, synth
        self.torch, self.ops, self._abi = torch, ops, _abi
        w = synth.QWEN32B_LAYER_M16384
        lins = {l.name: l for l in w.linears}
        self.x_attn = synth.activation(w, M32, H32, 0, dev)
        self.attn_out = synth.activation(w, M32, H32, 1, dev)
        self.x_mlp = synth.activation(w, M32, H32, 2, dev)
        self.gamma = torch.ones(H32, dtype=torch.bfloat16, device=dev)
        self.w = {n: synth.weight(w, lins[n], 10 + i, dev) for i, n in enumerate(LIN32)}
        # gradients of the linears' outputs; gate_up's comes from dH (the DGrad of down)
        # through the SiLU-mul backward inside the step
        self.dy = {n: synth.gradient(w, M32, LIN32[n][0], 20 + i, dev)
                   for i, n in enumerate(LIN32) if n != "gate_up"}
        self.eps = 1e-5
        # per-step batch tensors (the layer's input activations and the gradients of its
        # outputs); the BF16 weights and gamma are model state that stays on the device and
        # that the step itself re-quantizes, as the optimizer's updates would require
        self.inputs = ["x_attn", "attn_out", "x_mlp"] + [f"dy.{n}" for n in self.dy]
        # what a step hands back: the layer's output and the four weight gradients
        self.results = ["y"] + [f"dw_{n}" for n in LIN32]
        self.outputs = {}

    def tensor(self, name):
        if "." in name:
            d, k = name.split(".")
            return getattr(self, d)[k]
        return getattr(self, name)

    def run(self, marks=None):
        ops, V = self.ops, self._abi
        mark = _Marks(self.torch, marks)
        mark("start")
        qw = {}
        for n in LIN32:
            qw[n] = ops.quantize_128x128(self.w[n]); mark(f"wq_{n}")
        acts = {}
        q, s, qT, sT, _ = ops.rmsnorm_quant(self.x_attn, self.gamma, self.eps); mark("rmsnorm_quant_attn")
        acts["qkv"] = (q, s, qT, sT)
        qkv = ops.gemm_fwd(q, s, qw["qkv"][0], qw["qkv"][1]); mark("fwd_qkv")
        q, s, qT, sT = ops.quantize_1x128(self.attn_out, dual=True); mark("dq_attn_out")
        acts["o"] = (q, s, qT, sT)
        o = ops.gemm_fwd(q, s, qw["o"][0], qw["o"][1]); mark("fwd_o")
        q, s, qT, sT, _ = ops.rmsnorm_quant(self.x_mlp, self.gamma, self.eps); mark("rmsnorm_quant_mlp")
        acts["gate_up"] = (q, s, qT, sT)
        gu = ops.gemm_fwd(q, s, qw["gate_up"][0], qw["gate_up"][1]); mark("fwd_gate_up")
        acts["down"] = ops.silu_mul_quant(gu); mark("silu_mul_quant")
        q, s = acts["down"][0], acts["down"][1]
        y = ops.gemm_fwd(q, s, qw["down"][0], qw["down"][1]); mark("fwd_down")
        out = {"qkv": qkv, "o": o, "y": y}
        for n in ("down", "gate_up", "o", "qkv"):
            if n == "gate_up":
                # dY of gate_up = [dg | du] from its output and dH, quantized both ways
                qd, sd, qdT, sdT = ops.silu_mul_bwd_quant(gu, out["dx_down"]); mark("silu_mul_bwd_quant")
            else:
                qd, sd, qdT, sdT = ops.quantize_1x128(self.dy[n], dual=True); mark(f"dq_dy_{n}")
            out[f"dx_{n}"] = ops.gemm_dgrad(qd, sd, qw[n][2], qw[n][1]); mark(f"dgrad_{n}")
            out[f"dw_{n}"] = ops.gemm_wgrad(qdT, sdT, acts[n][2], acts[n][3]); mark(f"wgrad_{n}")
        self.outputs = out
        return out


class Mlp8Step:
    """Llama-3.1-8B MLP training step at 8192 tokens (forward, DGrad, WGrad, weight refresh)."""

    LAUNCHES_PER_STEP = 14

    def __init__(self, dev):
        import torch
        from block_scaled_fp8_x1_gb300 import _abi, ops, synth
        self.torch, self.ops, self._abi = torch, ops, _abi
        w = synth.LLAMA8B_MLP_M8192
        wb = synth.LLAMA8B_MLP_BWD_M8192
        gate_up, down = w.linears
        self.x = synth.activation(w, M_TOK, HID, 0, dev)
        self.gamma = torch.ones(HID, dtype=torch.bfloat16, device=dev)
        self.w_gu = synth.weight(w, gate_up, 1, dev)
        self.w_d = synth.weight(w, down, 2, dev)
        self.dy_d = synth.gradient(wb, M_TOK, HID, 3, dev)
        self.eps = w.extra["eps"]

    def run(self, marks=None):
        ops, V = self.ops, self._abi
        mark = _Marks(self.torch, marks)
        mark("start")
        q_gu, s_gu, qT_gu = ops.quantize_128x128(self.w_gu); mark("wq_gate_up")
        q_d, s_d, qT_d = ops.quantize_128x128(self.w_d); mark("wq_down")
        qx, sx, qxT, sxT, rstd = ops.rmsnorm_quant(self.x, self.gamma, self.eps); mark("rmsnorm_quant")
        gu = ops.gemm_fwd(qx, sx, q_gu, s_gu); mark("fwd_gate_up")
        qh, sh, qhT, shT = ops.silu_mul_quant(gu); mark("silu_mul_quant")
        y = ops.gemm_fwd(qh, sh, q_d, s_d); mark("fwd_down")
        qdy, sdy, qdyT, sdyT = ops.quantize_1x128(self.dy_d, dual=True); mark("dq_dy_down")
        dh = ops.gemm_dgrad(qdy, sdy, qT_d, s_d); mark("dgrad_down")
        dw_d = ops.gemm_wgrad(qdyT, sdyT, qhT, shT); mark("wgrad_down")
        # dY of gate_up = [dg | du] from its output and dH, quantized both ways
        qg, sg, qgT, sgT = ops.silu_mul_bwd_quant(gu, dh); mark("silu_mul_bwd_quant")
        dx = ops.gemm_dgrad(qg, sg, qT_gu, s_gu); mark("dgrad_gate_up")
        dw_gu = ops.gemm_wgrad(qgT, sgT, qxT, sxT); mark("wgrad_gate_up")
        return {"y": y, "dh": dh, "dx": dx, "dw_gu": dw_gu, "dw_d": dw_d}


def time_steps(step, steps, torch):
    """(ms per step over `steps` back-to-back steps, {kernel: [ms, ...]} from a second pass
    with an event after every launch)."""
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step.run()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return ms


def per_kernel(step, passes, torch):
    """Per-launch durations from events between launches.  Each pass starts on an idle
    device: a short device-side spin ahead of the first mark lets the host queue the whole
    step first, so that no interval holds host launch time."""
    per = {}
    for _ in range(passes):
        marks = []
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(8_000_000)   # about 4 ms at 2 GHz
        step.run(marks)
        torch.cuda.synchronize()
        for (_, a), (name, b) in zip(marks[:-1], marks[1:]):
            per.setdefault(name, []).append(a.elapsed_time(b))
    return {k: statistics.mean(v) for k, v in per.items()}


def kernel_table(per_ms, flops, qbytes, fp8_peak, hbm):
    kern = {}
    for name, ms in per_ms.items():
        e = {"ms": round(ms, 4)}
        if name in flops:
            tf = flops[name] / (ms * 1e-3) / 1e12
            e.update({"TFLOP/s": round(tf, 1), "frac_fp8_peak": round(tf / fp8_peak, 3)})
        elif name in qbytes:
            gbs = qbytes[name] / (ms * 1e-3) / 1e9
            e.update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)})
        kern[name] = e
    return kern


def backward_ops_table(dev, hbm, reps=10):
    """The operators either side of the gradient quantizer at the 32B layer's sizes (16384
    tokens): SiLU-mul backward into the dual-quantized gate_up gradient, RMSNorm backward,
    and the 128x1 WGrad operand re-quantized from a saved 1x128 activation.  Algorithmic
    HBM bytes per launch; times from CUDA events over `reps` back-to-back launches."""
    import torch
    from block_scaled_fp8_x1_gb300 import ops, synth
    M, H, I = M32, H32, LIN32["down"][1]
    rows = {}

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    gu = synth.normal_bf16((M, 2 * I), 2.0, 101, dev)
    dh = synth.normal_bf16((M, I), 1e-3, 102, dev)
    ms = timed(lambda: ops.silu_mul_bwd_quant(gu, dh))
    by = 2 * M * 2 * I + 2 * M * I + 2 * M * 2 * I + 8 * M * 2 * I / 128
    rows["silu_mul_bwd_quant"] = {"shape": [M, I], "ms": round(ms, 4), "GB/s": round(by / ms / 1e6, 1),
                                  "frac_hbm": round(by / ms / 1e6 / hbm, 3)}
    del gu, dh
    x = synth.normal_bf16((M, H), 1.0, 103, dev)
    dy = synth.normal_bf16((M, H), 1e-3, 104, dev)
    g = torch.ones(H, dtype=torch.bfloat16, device=dev)
    _, _, _, _, rstd = ops.rmsnorm_quant(x, g, 1e-5, dual=False)
    ms = timed(lambda: ops.rmsnorm_bwd(x, g, rstd, dy))
    by = 2 * 2 * M * H + 2 * M * H + 4 * M + 2 * H + 4 * H
    rows["rmsnorm_bwd"] = {"shape": [M, H], "ms": round(ms, 4), "GB/s": round(by / ms / 1e6, 1),
                           "frac_hbm": round(by / ms / 1e6 / hbm, 3)}
    for K in (H, I):
        xk = synth.normal_bf16((M, K), 1.0, 105, dev)
        q, sc = ops.quantize_1x128(xk)
        del xk
        ms = timed(lambda: ops.requantize_128x1(q, sc))
        by = 2 * M * K + 8 * M * K / 128
        rows[f"requantize_128x1_k{K}"] = {"shape": [M, K], "ms": round(ms, 4), "GB/s": round(by / ms / 1e6, 1),
                                          "frac_hbm": round(by / ms / 1e6 / hbm, 3)}
        del q, sc
    torch.cuda.empty_cache()
    return rows


def decode_table(dev, fp8_peak, hbm, reps=40, fmt="fp8"):
    """Qwen2.5-7B decode linears at M in {64, 128, 256}: the fused linear (activation
    quantization, then the decode GEMM) per call, timed as CUDA-graph replays of `reps` calls that cycle through
    weight copies larger than L2 in total, so every call streams its weights from HBM.
    fmt "fp8": the FP8 linear (1x128 activations, 128x128 weight blocks); "nvfp4": the NVFP4
    rollout linear (fp8_peak is then the FP4 peak).  Returns {"<linear>_m<M>": {...}} with
    the roofline fraction max(FLOP/peak, bytes/HBM) / time."""
    import torch
    from block_scaled_fp8_x1_gb300 import _abi, ops, synth
    w = synth.QWEN7B_DECODE
    lins = {l.name: l for l in w.linears}
    rows = {}
    for li, (name, (N, K)) in enumerate(DEC7B.items()):
        wb = synth.weight(w, lins[name], 30 + li, dev)
        if fmt == "nvfp4":
            wq = ops.quantize_nvfp4(wb)
            wbytes = N * K // 2
        else:
            wq = ops.quantize_128x128(wb, transpose=False)[:2]
            wbytes = N * K
        del wb
        ncopy = max(2, -(-(512 << 20) // wbytes))
        copies = [tuple(t.clone() for t in wq) for _ in range(ncopy)]
        del wq
        for M in DEC_M:
            x = synth.activation(w, M, K, 40 + li, dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

            def call(i):
                # the fused linear: quantization of x, then the decode GEMM overlapping it
                if fmt == "nvfp4":
                    ops.linear_nvfp4(x, *copies[i % ncopy], out=y)
                else:
                    ops.linear_fwd(x, copies[i % ncopy][0], copies[i % ncopy][1], out=y)

            for i in range(3):
                call(i)
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    for i in range(reps):
                        call(i)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (5 * reps)
            fl, by = (decode_work_nvfp4 if fmt == "nvfp4" else decode_work)(M, N, K)
            roof_us = max(fl / (fp8_peak * 1e12), by / (hbm * 1e9)) * 1e6
            rows[f"{name}_m{M}"] = {"M": M, "N": N, "K": K, "us": round(us, 2),
                                    "GB/s": round(by / (us * 1e-6) / 1e9, 1),
                                    "TFLOP/s": round(fl / (us * 1e-6) / 1e12, 1),
                                    "roofline_us": round(roof_us, 2),
                                    "frac_roofline": round(roof_us / us, 3)}
            del g, x, y
        del copies
        torch.cuda.empty_cache()
    return rows


def max_over_ranks(ms: float, device) -> float:
    """The largest of every rank's time (the job ends when its slowest replica does); the
    time itself with a single rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the work every replica did, over the slowest replica's time
    (work units per second)."""
    return work_per_rank * world / (ms * 1e-3)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_scaled_fp8_x1_gb300 import build_library, ops
    build_library()
    ops.init(local)

    peaks = measured_peaks()
    # kernels are timed inside a sub-second region: the burst rate is their ceiling
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    hbm = peaks["hbm_gbs"]

    step = Layer32Step(dev)
    flops, qbytes = layer32_work()
    step_flops = sum(flops.values())

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step.run()
    barrier()

    # ---- device-resident timed region: whole steps
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    w0 = time.time()
    ms_total = time_steps(step, args.steps, torch)
    barrier()
    w1 = time.time()
    clk = clocks.stop((w0, w1))
    ms_step = max_over_ranks(ms_total, dev)
    # per-kernel split (separate passes, same work)
    per = per_kernel(step, max(3, min(args.steps, 10)), torch)
    st = ops.check_status()

    # ---- end to end: host buffers, copies inside the timed region.  Every step uploads
    # its inputs from pinned host memory and downloads its results; the copies run on two
    # copy streams and overlap the neighbouring steps' compute (two device input sets,
    # ordered by events), as a training loop that feeds the GPU would.
    host_in = {n: torch.empty_like(step.tensor(n), device="cpu").pin_memory() for n in step.inputs}
    for n in step.inputs:
        host_in[n].copy_(step.tensor(n))
    outs = step.run()
    host_out = {k: torch.empty_like(outs[k], device="cpu").pin_memory() for k in step.results}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    sets = [step, Layer32Step(dev)]               # device input sets, used alternately
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    uploaded = [torch.cuda.Event(), torch.cuda.Event()]
    computed = [torch.cuda.Event(), torch.cuda.Event()]
    for e in computed:
        e.record(comp)

    def upload(i):
        sset = sets[i % 2]
        up.wait_event(computed[i % 2])            # the set's previous step is done with it
        with torch.cuda.stream(up):
            for n in sset.inputs:
                sset.tensor(n).copy_(host_in[n], non_blocking=True)
        uploaded[i % 2].record(up)

    def compute_and_download(i):
        comp.wait_event(uploaded[i % 2])
        o = sets[i % 2].run()
        computed[i % 2].record(comp)
        down.wait_event(computed[i % 2])
        with torch.cuda.stream(down):
            for k in host_out:
                o[k].record_stream(down)
                host_out[k].copy_(o[k], non_blocking=True)

    def e2e_steps(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute_and_download(i)
        comp.wait_stream(down)

    e2e_steps(max(1, args.warmup))
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    up.wait_event(e0)
    down.wait_event(e0)
    e2e_steps(args.steps)
    e1.record(comp)
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    del sets, host_in, host_out, outs
    step.outputs = {}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    kern = kernel_table(per, flops, qbytes, fp8_peak, hbm)
    dominant = max(kern, key=lambda n: kern[n]["ms"])
    dom_ms = kern[dominant]["ms"]
    if dominant in flops:
        achieved = flops[dominant] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 3),
                "traffic": load_traffic(dominant), "kernel": dominant,
                "frac_of_nominal_4500": round(achieved / FP8_NOMINAL_TFLOPS, 3),
                "peak_note": f"{peaks['source']} burst bf16 {peaks['bf16_tflops']} x {FP8_PER_BF16} "
                             f"(nominal FP8/BF16 ratio); kernels timed in a sub-second region"}
    else:
        achieved = qbytes[dominant] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 3), "traffic": load_traffic(dominant),
                "kernel": dominant, "peak_note": f"{peaks['source']} copy bandwidth"}
    value = job_rate(step_flops, world, ms_step) / 1e12

    # ---- beside the headline: the 8B MLP step and the 7B decode linears (rank 0 only)
    extra = {}
    if not args.no_extra:
        torch.cuda.empty_cache()
        s8 = Mlp8Step(dev)
        f8, b8 = mlp8_work()
        for _ in range(3):
            s8.run()
        torch.cuda.synchronize()
        ms8 = time_steps(s8, args.steps, torch)
        k8 = kernel_table(per_kernel(s8, 5, torch), f8, b8, fp8_peak, hbm)
        extra["llama8b_mlp_step"] = {
            "workload": "Llama-3.1-8B MLP training step at 8192 tokens (gate_up 28672x4096, "
                        "down 4096x14336; fwd + DGrad + WGrad, weight refresh; dY of gate_up "
                        "from dH through the SiLU-mul backward)",
            "ms_per_step": round(ms8, 4), "TFLOP/s": round(sum(f8.values()) / (ms8 * 1e-3) / 1e12, 1),
            "kernels": k8}
        del s8
        torch.cuda.empty_cache()
        extra["qwen7b_decode"] = decode_table(dev, fp8_peak, hbm)
        extra["qwen7b_decode_nvfp4"] = decode_table(dev, 3.0 * fp8_peak, hbm, fmt="nvfp4")
        extra["backward_ops_32b"] = backward_ops_table(dev, hbm)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": M32, "hidden": H32,
                   "linears": {k: list(v) for k, v in LIN32.items()},
                   "gemm_flops_per_step": step_flops,
                   "l2": "inputs larger than L2 (X 168 MB each, W_gate_up 566 MB, gate_up output 1.8 GB per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "e2e": {"value": round(job_rate(step_flops, world, ms_e2e) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4),
                "copies": "every step's batch tensors (X_attn, attention output, X_mlp, the dY of qkv, o and down) up from pinned host memory and its results (y, the four dW) down, on two copy streams overlapping the neighbouring steps' compute; the BF16 weights stay on the device as model state and are re-quantized by the step"},
        "gpu_launches": Layer32Step.LAUNCHES_PER_STEP * args.steps,
        "clocks": clk,
        "kernels": kern,
        "device_status": st,
    }
    line.update(extra)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


GEMM_SOURCES = ("block_scaled_fp8_x1_gb300/csrc/gemm.cu", "block_scaled_fp8_x1_gb300/csrc/gemm_tiled.cuh",
                "block_scaled_fp8_x1_gb300/csrc/gemm_pair.cu", "block_scaled_fp8_x1_gb300/csrc/common.cuh",
                "block_scaled_fp8_x1_gb300/csrc/gemm.h")


def gemm_sources_hash() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when that capture was taken on other GEMM sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        if d.get("gemm_sources_sha256_16") != gemm_sources_hash():
            return None
        e = d.get(kernel)
        return e["bytes_per_launch"] if e else None
    except Exception:
        return None


# ----------------------------------------------------------------------------- oracle arm

def oracle_step_estimate(rows: int, n_samp: int):
    """Time the CPU oracle on a bounded sample of every kernel of the 32B layer step
    (quantizers on `rows` token rows or weight rows, GEMMs on `n_samp` output elements) and
    extrapolate each to its full size.  Returns (estimated seconds for one full step,
    threads, sample description)."""
    import numpy as np
    import torch

    import oracle
    from block_scaled_fp8_x1_gb300 import synth

    threads = oracle.threads()
    w = synth.QWEN32B_LAYER_M16384
    lins = {l.name: l for l in w.linears}
    rng = np.random.default_rng(0)

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def timed(fn):
        t = time.perf_counter()
        out = fn()
        return time.perf_counter() - t, out

    est = 0.0
    x = bits(synth.activation(w, rows, H32, 0))
    gamma = np.full(H32, 0x3F80, np.uint16)
    # weight refresh: 128 weight rows of each linear, scaled by its rows
    for n, (N, K) in LIN32.items():
        wb = bits(synth.normal_bf16((128, K), w.weight_std, 7))
        t, _ = timed(lambda: oracle.quantize_128x128(wb))
        est += t * N / 128
    # two RMSNorm dual quantizers, the attention-output dual quantizer
    t, r = timed(lambda: oracle.rmsnorm_quant(x, gamma, 1e-5))
    est += 2 * t * M32 / rows
    t, _ = timed(lambda: (oracle.quantize_1x128(x), oracle.quantize_128x1(x)))
    est += t * M32 / rows
    # SiLU-mul on the gate_up output, then its dual quantization
    I = LIN32["down"][1]
    gu = bits(synth.normal_bf16((rows, 2 * I), 2.0, 9))
    t, h = timed(lambda: oracle.silu_mul(gu))
    t2, _ = timed(lambda: (oracle.quantize_1x128(h[0]), oracle.quantize_128x1(h[0])))
    est += (t + t2) * M32 / rows
    # dual quantization of the dY of qkv, o and down, per element of the sampled rows
    t, _ = timed(lambda: (oracle.quantize_1x128(x), oracle.quantize_128x1(x)))
    est += t * M32 / rows * sum(N for n, (N, _) in LIN32.items() if n != "gate_up") / H32
    # the SiLU-mul backward of gate_up with the dual quantization of [dg | du]
    dh = bits(synth.normal_bf16((rows, I), 1e-3, 10))
    t, _ = timed(lambda: oracle.silu_mul_bwd_quant(gu, dh))
    est += t * M32 / rows
    parts = [f"quantizers on {rows} token rows / 128 weight rows"]
    # GEMMs: sampled output elements, scaled by outputs / samples
    qx, sx = r[0], r[1]
    qw, sw, _ = oracle.quantize_128x128(bits(synth.weight(w, lins["qkv"], 1)[:256]))
    i1 = rng.integers(0, rows, n_samp)
    i2 = rng.integers(0, 256, n_samp)
    t, _ = timed(lambda: oracle.gemm_sampled(qx, sx, qw, sw, "fwd", i1, i2))
    per_flop = t / (2.0 * H32 * n_samp)
    f, _ = layer32_work()
    est += per_flop * sum(f.values())
    parts.append(f"{n_samp} GEMM outputs (K={H32}) extrapolated per FLOP")
    return est, threads, "; ".join(parts)


def cpu_baseline():
    est, threads, sample = oracle_step_estimate(rows=512, n_samp=4096)
    f, _ = layer32_work()
    flops = sum(f.values())
    return {"value": round(flops / est / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": sample + f"; full step extrapolated to {est:.1f} s",
            "ms_per_step_extrapolated": round(est * 1e3, 1)}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle_step_estimate(rows=256, n_samp=1024)
    ests = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e, threads, sample = oracle_step_estimate(rows=256, n_samp=1024)
        ests.append(e)
    wall = time.perf_counter() - t0
    est = statistics.median(ests)
    f, _ = layer32_work()
    flops = sum(f.values())
    value = flops / est / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(est * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle: binary64 block sums, binary32 quantizers)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": M32, "hidden": H32,
                   "linears": {k: list(v) for k, v in LIN32.items()}},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample + f"; {args.steps} samples in {wall:.1f} s"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_kernel(args):
    """One kernel form on one shape, `reps` launches after one warm-up, with CUDA-event
    timing (used for ncu captures on small cases and for kernel sweeps)."""
    import torch
    from block_scaled_fp8_x1_gb300 import _abi, build_library, ops, synth
    build_library()
    ops.init(0)
    dev = torch.device("cuda", 0)
    dims = [int(v) for v in args.shape.split(",")]
    k = args.kernel
    if k.startswith("gemm"):
        M, N, K = dims
        var = {"auto": _abi.FP8RL_VARIANT_AUTO, "tiled": _abi.FP8RL_VARIANT_TILED,
               "pair": _abi.FP8RL_VARIANT_PAIR, "decode": _abi.FP8RL_VARIANT_DECODE}[args.variant]
        if k == "gemm_wgrad":
            a = ops.quantize_128x1(synth.normal_bf16((M, N), 1e-3, 1, dev))
            b = ops.quantize_128x1(synth.normal_bf16((M, K), 1.0, 2, dev))
            fn = lambda: ops.gemm_wgrad(a[0], a[1], b[0], b[1], variant=var, epi_warps=args.epi, tile_n=args.tile_n)
        else:
            lhs_cols = N if k == "gemm_dgrad" else K
            qa, sa = ops.quantize_1x128(synth.normal_bf16((M, lhs_cols), 1.0, 1, dev))
            if k == "gemm_dgrad":
                _, sw, qwT = ops.quantize_128x128(synth.normal_bf16((N, K), 0.02, 2, dev))
                fn = lambda: ops.gemm_dgrad(qa, sa, qwT, sw, variant=var, epi_warps=args.epi, tile_n=args.tile_n)
            else:
                qw, sw, _ = ops.quantize_128x128(synth.normal_bf16((N, K), 0.02, 2, dev), transpose=False)
                if k == "gemm_decode":
                    var = _abi.FP8RL_VARIANT_DECODE if args.variant == "decode" else _abi.FP8RL_VARIANT_SPLITK
                # decode streams each layer's weights once: cycle through copies that together
                # exceed L2 so that back-to-back launches read HBM, not L2
                ncopy = max(1, -(-(256 << 20) // (N * K))) if k == "gemm_decode" else 1
                ws = [(qw.clone(), sw.clone()) for _ in range(ncopy)] if ncopy > 1 else [(qw, sw)]
                it = [0]

                def fn():
                    w_q, w_s = ws[it[0] % len(ws)]
                    it[0] += 1
                    return ops.gemm_fwd(qa, sa, w_q, w_s, variant=var, tile_n=args.tile_n,
                                        epi_warps=args.epi)
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif k == "nvfp4_decode":                # shape M,N,K: the NVFP4 GEMM alone, GB/s of its bytes
        M, N, K = dims
        xq = ops.quantize_nvfp4(synth.normal_bf16((M, K), 1.0, 1, dev))
        wq = ops.quantize_nvfp4(synth.normal_bf16((N, K), 0.02, 2, dev))
        ncopy = max(1, -(-(256 << 20) // (N * K // 2)))
        ws = [tuple(t.clone() for t in wq) for _ in range(ncopy)]
        it = [0]

        def fn():
            w = ws[it[0] % len(ws)]
            it[0] += 1
            return ops.gemm_nvfp4(*xq, *w)
        work = N * K // 2 + N * K // 16 + 4 * N + M * K // 2 + M * K // 16 + 2 * M * N
        unit = "GB/s"
    else:
        M, K = dims
        if k == "rmsnorm_quant":
            x = synth.normal_bf16((M, K), 1.0, 1, dev)
            g = torch.ones(K, dtype=torch.bfloat16, device=dev)
            fn = lambda: ops.rmsnorm_quant(x, g, 1e-5)
            work = M * K * (2 + 2) + 8 * M * K / 128
        elif k == "silu_mul_quant":
            x = synth.normal_bf16((M, 2 * K), 1.0, 1, dev)
            fn = lambda: ops.silu_mul_quant(x)
            work = M * K * (4 + 2) + 8 * M * K / 128
        elif k == "quant_dual":
            x = synth.normal_bf16((M, K), 1.0, 1, dev)
            fn = lambda: ops.quantize_1x128(x, dual=True)
            work = M * K * (2 + 2) + 8 * M * K / 128
        elif k == "quant_128x128":
            x = synth.normal_bf16((M, K), 0.02, 1, dev)
            fn = lambda: ops.quantize_128x128(x)
            work = M * K * (2 + 2) + 4 * M * K / 16384
        elif k == "rmsnorm_bwd":
            x = synth.normal_bf16((M, K), 1.0, 1, dev)
            dy = synth.normal_bf16((M, K), 1e-3, 2, dev)
            g = torch.ones(K, dtype=torch.bfloat16, device=dev)
            _, _, _, _, rstd = ops.rmsnorm_quant(x, g, 1e-5, dual=False)
            fn = lambda: ops.rmsnorm_bwd(x, g, rstd, dy)
            work = M * K * (2 + 2 + 2) + 4 * M + 2 * K + 4 * K
        elif k == "silu_mul_bwd_quant":      # shape M,I: gu [M,2I], dh [M,I]
            gu = synth.normal_bf16((M, 2 * K), 2.0, 1, dev)
            dh = synth.normal_bf16((M, K), 1e-3, 2, dev)
            fn = lambda: ops.silu_mul_bwd_quant(gu, dh)
            work = 2 * M * 2 * K + 2 * M * K + 2 * M * 2 * K + 8 * M * 2 * K / 128
        elif k == "quant_nvfp4":
            x = synth.normal_bf16((M, K), 0.02, 1, dev)
            fn = lambda: ops.quantize_nvfp4(x)
            work = M * K * 2 + M * K // 2 + M * K // 16 + 4 * M
        elif k == "requantize_128x1":
            q, s = ops.quantize_1x128(synth.normal_bf16((M, K), 1.0, 1, dev))
            fn = lambda: ops.requantize_128x1(q, s)
            work = M * K * (1 + 1) + 8 * M * K / 128
        else:
            raise SystemExit(f"unknown kernel {k}")
        unit = "GB/s"
    fn()
    torch.cuda.synchronize()
    # launches queued back to back between two events, so that the host's per-call work
    # (argument checks, tensor-map encoding) overlaps the device time of earlier launches
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.reps):
        fn()
    ev1.record()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / args.reps
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"kernel": k, "shape": dims, "ms": round(ms, 4), unit: round(rate, 1),
                      "status": ops.check_status()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 8B MLP step and the 7B decode table beside the headline")
    ap.add_argument("--kernel", default=None,
                    help="run one kernel form alone (for profiling): gemm_fwd, gemm_dgrad, "
                         "gemm_wgrad, gemm_decode, rmsnorm_quant, silu_mul_quant, quant_dual, "
                         "quant_128x128, rmsnorm_bwd, silu_mul_bwd_quant, requantize_128x1, "
                         "quant_nvfp4, nvfp4_decode")
    ap.add_argument("--shape", default=None, help="M,N,K (GEMMs) or M,K (quantizers)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--tile-n", type=int, default=0, help="GEMM tile width (128/256) of the tiled or paired form")
    ap.add_argument("--variant", default="auto", choices=["auto", "tiled", "pair", "decode"],
                    help="GEMM form for --kernel gemm_fwd/gemm_dgrad/gemm_wgrad; gemm_decode: "
                         "decode (weights on the MMA's M side) or the split-K form (default)")
    ap.add_argument("--epi", type=int, default=0, help="paired form: epilogue warps per CTA (8/16)")
    args = ap.parse_args()
    if args.kernel:
        run_kernel(args)
        return
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
