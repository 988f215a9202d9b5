"""Host-side measurement logic of bench.py (CPU only).

The algorithmic byte counts are the ones the roofline divides by: weights +
bf16 activations + bf16 outputs per launch, for the decode shapes (4096,
4096), (14336, 4096), (4096, 14336) and the NVFP4 N = K = 4096 case.  The
expected numbers are written out from the format definitions (one byte per
E4M3 code, half a byte per E2M1 code, one E4M3 scale per 16 elements, two
bytes per bf16 value), not from the functions under test.
"""

import hashlib
import json
import os
import shutil

import pytest

import bench


@pytest.mark.parametrize("n,k,want", [(4096, 4096, 16_793_600), (14336, 4096, 58_757_120),
                                      (4096, 14336, 58_757_120), (256, 520, 134_672)])
def test_fp8_gemv_algorithmic_bytes(n, k, want):
    assert bench.fp8_gemv_bytes(n, k) == want == n * k + 2 * k + 2 * n


@pytest.mark.parametrize("m,want", [(1, 9_453_568), (16, 9_699_328), (128, 11_534_336)])
def test_nvfp4_algorithmic_bytes(m, want):
    n = k = 4096
    assert bench.nvfp4_bytes(m, n, k) == want == n * k // 2 + n * k // 16 + 2 * m * k + 2 * m * n


@pytest.mark.parametrize("set_bytes", [1, 16_793_600, 134_307_840, 470_000_000, 10**10])
def test_weight_rotation_defeats_l2(set_bytes):
    copies = bench.n_copies(set_bytes)
    assert copies >= 2
    if set_bytes * 2 < bench.ROTATION_TARGET:
        assert copies * set_bytes >= bench.ROTATION_TARGET >= 4 * bench.L2_BYTES


def test_committed_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src_rel = os.path.join("gemm_fp8_nvfp4_gb300", "csrc", "gemv.cu")
    (tmp_path / "gemm_fp8_nvfp4_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, src_rel), tmp_path / src_rel)
    h = hashlib.sha256(open(tmp_path / src_rel, "rb").read()).hexdigest()[:16]
    entry = {"kernel": "k", "source": src_rel, "source_sha256_16": h, "bytes_per_launch": 123}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"fp8_gemv": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("fp8_gemv") == 123
    assert bench.committed_traffic("other_kernel") is None
    # any change to the kernel source voids the figure
    with open(tmp_path / src_rel, "a") as f:
        f.write("\n// changed\n")
    assert bench.committed_traffic("fp8_gemv") is None


def test_committed_traffic_file_is_well_formed():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for ent in d.values():
        assert os.path.exists(os.path.join(bench.ROOT, ent["source"]))
        assert len(ent["source_sha256_16"]) == 16 and ent["bytes_per_launch"] > 0


@pytest.mark.parametrize("bytes_per_copy", [
    14336 * 4096 + 2 * 2048 * 4096,    # FP8 / W8A8 GEMM M = 2048: weights + activations
    14336 * 4100 + 2 * 2048 * 4100,    # any-K GEMM
    2 * 2048 * 4096,                   # W8A8 quantizer: the activations alone
    1, 3 * bench.L2_BYTES])
def test_sub_benchmark_rotation_exceeds_l2(bytes_per_copy):
    copies = bench.copies_past_l2(bytes_per_copy)
    assert copies >= 2
    assert copies * bytes_per_copy >= 2 * bench.L2_BYTES
