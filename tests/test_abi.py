"""The C-ABI library builds, loads without a GPU and exports every symbol
that include/gq.h declares (no compute calls: there may be no GPU here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    from gemm_fp8_nvfp4_gb300 import _build
    if not os.path.exists(_build.LIB):
        _build.build()
    return _build.LIB


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("gq_fp8_gemv", "gq_fp8_matmul", "gq_fp8_grouped_matmul", "gq_nvfp4_gemv",
                 "gq_nvfp4_matmul", "gq_fp8_materialize", "gq_nvfp4_materialize",
                 "gq_status_str"):
        assert name in syms, name


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in gq.h but not exported"


def test_binding_declares_every_symbol(lib_path):
    import gemm_fp8_nvfp4_gb300 as gq
    assert sorted(gq.SIGNATURES) == declared_symbols()
    lib = gq.load_library(lib_path)
    assert lib.gq_version().decode().startswith("gq ")


def test_status_strings(lib_path):
    import gemm_fp8_nvfp4_gb300 as gq
    gq.load_library(lib_path)
    for s in range(9):
        assert gq.status_str(s).startswith("GQ_")
    assert "unknown" in gq.status_str(99)


def test_library_has_no_runtime_link_to_cuda_driver_or_torch(lib_path):
    """The library must load on a machine without libcuda (this one) and must
    not depend on torch: check its dynamic dependencies."""
    import subprocess
    out = subprocess.run(["ldd", lib_path], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out
    assert "libtorch" not in out and "libc10" not in out
    assert "not found" not in out


def test_product_package_never_touches_the_oracle():
    """The product code (binding + CUDA sources) imports nothing from oracle/."""
    pkg = os.path.join(ROOT, "gemm_fp8_nvfp4_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("no oracle", ""), os.path.join(dirpath, f)


def test_every_op_refuses_host_tensors():
    """The product path has no CPU fallback: every op given host tensors
    raises before anything runs (nothing is computed off the GPU)."""
    import torch

    import gemm_fp8_nvfp4_gb300 as gq

    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    u8 = lambda *s: torch.zeros(*s, dtype=torch.uint8)
    i8 = lambda *s: torch.zeros(*s, dtype=torch.int8)
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32)
    k = 64
    calls = {
        "fp8_gemv": lambda: gq.fp8_gemv(bf(k), u8(8, k), 1.0),
        "nvfp4_gemv": lambda: gq.nvfp4_gemv(bf(k), u8(8, k // 2), u8(8, k // 16), 1.0),
        "fp8_matmul": lambda: gq.fp8_matmul(bf(4, k), u8(8, k), 1.0),
        "nvfp4_matmul": lambda: gq.nvfp4_matmul(bf(4, k), u8(8, k // 2), u8(8, k // 16), 1.0),
        "fp8_grouped_matmul": lambda: gq.fp8_grouped_matmul(
            bf(4, k), u8(2, 8, k), i32(3), i32(2), max_rows_per_group=4),
        "nvfp4_grouped_matmul": lambda: gq.nvfp4_grouped_matmul(
            bf(4, k), u8(2, 8, k // 2), u8(2, 8, k // 16), i32(3), i32(2), max_rows_per_group=4),
        "int8_quantize_rows": lambda: gq.int8_quantize_rows(bf(4, k)),
        "int8_matmul": lambda: gq.int8_matmul(i8(4, k), i8(8, k), f32(4), f32(8)),
        "fp8_materialize": lambda: gq.fp8_materialize(u8(8, k)),
        "nvfp4_materialize": lambda: gq.nvfp4_materialize(u8(8, k // 2), u8(8, k // 16)),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def test_every_op_refuses_tensors_of_another_device(monkeypatch):
    """The library launches on the current device: operands, outputs and
    streams of another GPU are refused in the binding before any launch.
    Checked on the CPU with tensors that claim to live on cuda:1 while
    cuda:0 is current (no GPU is touched)."""
    import torch

    import gemm_fp8_nvfp4_gb300 as gq

    monkeypatch.setattr(gq, "_current_device_index", lambda: 0)

    class OnCuda1(torch.Tensor):
        @property
        def is_cuda(self):
            return True

        @property
        def device(self):
            return torch.device("cuda", 1)

    def far(t):
        return torch.Tensor._make_subclass(OnCuda1, t)

    bf = lambda *s: far(torch.zeros(*s, dtype=torch.bfloat16))
    u8 = lambda *s: far(torch.zeros(*s, dtype=torch.uint8))
    i8 = lambda *s: far(torch.zeros(*s, dtype=torch.int8))
    f32 = lambda *s: far(torch.zeros(*s, dtype=torch.float32))
    i32 = lambda *s: far(torch.zeros(*s, dtype=torch.int32))
    k = 64
    calls = {
        "fp8_gemv": lambda: gq.fp8_gemv(bf(k), u8(8, k), 1.0),
        "nvfp4_gemv": lambda: gq.nvfp4_gemv(bf(k), u8(8, k // 2), u8(8, k // 16), 1.0),
        "fp8_matmul": lambda: gq.fp8_matmul(bf(4, k), u8(8, k), 1.0),
        "nvfp4_matmul": lambda: gq.nvfp4_matmul(bf(4, k), u8(8, k // 2), u8(8, k // 16), 1.0),
        "fp8_grouped_matmul": lambda: gq.fp8_grouped_matmul(
            bf(4, k), u8(2, 8, k), i32(3), i32(2), max_rows_per_group=4),
        "nvfp4_grouped_matmul": lambda: gq.nvfp4_grouped_matmul(
            bf(4, k), u8(2, 8, k // 2), u8(2, 8, k // 16), i32(3), i32(2), max_rows_per_group=4),
        "int8_quantize_rows": lambda: gq.int8_quantize_rows(bf(4, k)),
        "int8_matmul": lambda: gq.int8_matmul(i8(4, k), i8(8, k), f32(4), f32(8)),
        "fp8_materialize": lambda: gq.fp8_materialize(u8(8, k)),
        "nvfp4_materialize": lambda: gq.nvfp4_materialize(u8(8, k // 2), u8(8, k // 16)),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="current device is cuda:0"):
            call()

    # a stream of another device is refused too; the current device passes
    class FakeStream:
        def __init__(self, index):
            self.device = torch.device("cuda", index)
            self.cuda_stream = 0

    with pytest.raises(ValueError, match="stream is on cuda:1"):
        gq._stream_handle(FakeStream(1))
    assert gq._stream_handle(FakeStream(0)) == 0
    gq._same_device(torch.device("cuda", 0), "x")


def test_launch_flags_accept_the_test_stall_bit_only_as_declared(lib_path):
    """gq_set_launch_flags takes GQ_LAUNCH_OVERLAP_WEIGHT_READS and
    GQ_LAUNCH_TEST_STALL_PRODUCER (host state only, no GPU needed) and
    refuses any other bit."""
    import gemm_fp8_nvfp4_gb300 as gq
    lib = gq.load_library(lib_path)
    assert gq.GQ_LAUNCH_TEST_STALL_PRODUCER == 2
    text = open(HEADER).read()
    assert "#define GQ_LAUNCH_TEST_STALL_PRODUCER 2u" in text
    try:
        assert lib.gq_set_launch_flags(2) == 0 and lib.gq_get_launch_flags() == 2
        assert lib.gq_set_launch_flags(3) == 0 and lib.gq_get_launch_flags() == 3
        assert lib.gq_set_launch_flags(4) == 2 and lib.gq_get_launch_flags() == 3
    finally:
        assert lib.gq_set_launch_flags(0) == 0
