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
