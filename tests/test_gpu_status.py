"""Failure detection without a GPU fault: a bounded device wait runs out, the kernel records
FP8RL_ERR_DEVICE_TIMEOUT in the status word and returns; the host reads and clears it and
the context stays usable."""
import pytest
import torch

from block_scaled_fp8_x1_gb300 import _abi, synth

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared(fp8lib):
    assert fp8lib.check_status() == _abi.FP8RL_OK
    fp8lib.debug_wait_timeout(5_000_000)            # 5 ms on a barrier nothing completes
    assert fp8lib.check_status() == _abi.FP8RL_ERR_DEVICE_TIMEOUT
    assert fp8lib.check_status() == _abi.FP8RL_OK   # read-and-clear
    # the context still works
    x = synth.normal_bf16((256, 512), 1.0, 1, "cuda")
    w = synth.normal_bf16((512, 512), 0.02, 2, "cuda")
    qx, sx = fp8lib.quantize_1x128(x)
    qw, sw, _ = fp8lib.quantize_128x128(w)
    y = fp8lib.gemm_fwd(qx, sx, qw, sw, variant=_abi.FP8RL_VARIANT_TILED)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    assert fp8lib.check_status() == _abi.FP8RL_OK


def test_argument_errors_raise(fp8lib):
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_abi.Fp8rlError) as e:
        fp8lib.quantize_1x128(x)
    assert e.value.status == _abi.FP8RL_ERR_SHAPE
