"""Shared pytest configuration: the ``gpu`` marker and repo-root imports."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(autouse=True, scope="module")
def _device_status_clean(request):
    """After every GPU test module: no bounded in-kernel wait of this process
    ran out (the per-device status word is 0; the time-out tests reset what
    they provoke)."""
    yield
    marks = getattr(request.module, "pytestmark", [])
    marks = marks if isinstance(marks, list) else [marks]
    if not any(getattr(m, "name", "") == "gpu" for m in marks):
        return
    import torch
    if not torch.cuda.is_available():
        return
    import gemm_fp8_nvfp4_gb300 as gq
    assert gq.device_status() == 0, "a bounded in-kernel wait ran out during this module"
