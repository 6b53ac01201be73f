"""Shared test setup: markers, library builds and GPU availability."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the CUDA library")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def oracle():
    import oracle as orc
    orc.build()
    return orc


@pytest.fixture(scope="session")
def fp8lib():
    """The CUDA library (built if stale).  GPU tests only."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    from block_scaled_fp8_x1_gb300 import build_library, ops
    build_library()
    ops.init(0)
    # a healthy kernel never waits this long on one barrier; fail fast instead of hanging
    ops.set_wait_timeout_ns(int(float(os.environ.get("FP8RL_TEST_WAIT_NS", "1e9"))))
    return ops
