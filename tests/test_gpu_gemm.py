"""tcgen05 GEMMs (FP8 and NVFP4) against the oracle.

Tolerance: |gpu - oracle| <= 2e-4 * |alpha| * sum_k |a_k w_k| (+1 bf16 ulp for
bf16 outputs).  The identity-activation tests check the in-kernel dequant of
every code exactly: with A = I the product returns the decoded weight itself.
"""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import (DEV, assert_canary, assert_exact, assert_within, bits, canary_out,
                            lib, to_f64)

pytestmark = pytest.mark.gpu


def check_fp8(m, n, k, out_dtype=torch.float32, seed=0, rows=None, alpha_mode="scale"):
    codes, scale = synth.fp8_weight(n, k, seed=seed)
    a = synth.bf16_activations(m, k, seed=seed + 1)
    alpha = scale if alpha_mode == "scale" else 1.0
    buf, c = canary_out((m, n), out_dtype)
    gq.fp8_matmul(a.to(DEV), codes.to(DEV), alpha, out=c)
    torch.cuda.synchronize()
    assert_canary(buf)
    got = to_f64(c)
    sel = np.arange(m) if rows is None else np.asarray(rows)
    ab = bits(a)[sel]
    w_hat = oracle.decode_fp8(codes.numpy())
    ref = oracle.linear(ab, w_hat, alpha)
    tol = oracle.tolerance(ab, w_hat, alpha, out_dtype == torch.bfloat16, ref=ref)
    assert_within(got[sel], ref, tol, f"fp8 gemm {m}x{n}x{k}")
    return c


@pytest.mark.parametrize("m,n,k", [(1, 256, 64), (128, 256, 64), (200, 384, 256), (3, 127, 16),
                                   (17, 257, 32), (129, 520, 112), (300, 1000, 4112),
                                   (64, 8, 1024), (2, 3, 48)])
def test_fp8_gemm_shapes(m, n, k):
    lib()
    check_fp8(m, n, k, seed=m + n + k)


# M > 128 runs on CTA pairs: tiles of 512 rows (each CTA of the pair holds
# rows 256 h + 128 rank + [0, 128) of the tile) and 256 weight rows (128 per
# CTA).  Row counts around 256 and 512, and N with the odd CTA's weight rows
# partly or wholly past the end.
PAIR_EDGES = [(129, 256, 64), (256, 200, 64), (257, 129, 128), (511, 300, 192), (512, 128, 64),
              (513, 384, 64), (1000, 520, 256), (1537, 260, 128)]


@pytest.mark.parametrize("m,n,k", PAIR_EDGES)
def test_fp8_gemm_pair_tile_edges(m, n, k):
    lib()
    check_fp8(m, n, k, seed=m + 2 * n + k)


@pytest.mark.parametrize("m,n,k", PAIR_EDGES)
def test_nvfp4_gemm_pair_tile_edges(m, n, k):
    lib()
    check_nvfp4(m, n, k, seed=m + 3 * n + k)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_gemm_bf16_and_f32_out(out_dtype):
    lib()
    check_fp8(256, 512, 512, out_dtype)


def test_fp8_gemm_prefill_config_sampled():
    """The M=2048, N=14336, K=4096 prefill GEMM in the benchmark's launch
    configuration; the oracle checks 48 rows (first, last, tile edges, random)."""
    lib()
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 1, 127, 128, 255, 1023, 2046, 2047] + list(rng.integers(0, 2048, 40))))
    check_fp8(2048, 14336, 4096, torch.bfloat16, seed=0, rows=rows)


def test_fp8_gemm_identity_dequant_every_code():
    """A = I: C[m, n] = w_hat[n, m] exactly (f32 out, alpha 1), for every E4M3 code
    including the NaN codes, through the tensor-core dequant path.  The result
    is a sum 1 * w + 0 * (others), so a -0 weight may come back as +0."""
    lib()
    k = 256
    codes = (np.arange(300 * k).reshape(300, k) * 7 % 256).astype(np.uint8)
    eye = torch.eye(k, dtype=torch.bfloat16)
    c = gq.fp8_matmul(eye.to(DEV), torch.from_numpy(codes).to(DEV), 1.0, out_dtype=torch.float32)
    got = to_f64(c)
    want = oracle.fp8_materialize(codes).T
    # NaN rows: any column hitting a NaN code is NaN in that row (0 * NaN = NaN)
    want = want.copy()
    nan_cols = np.isnan(oracle.fp8_materialize(codes)).any(axis=1)
    want[:, nan_cols] = np.nan
    assert_exact(got, want, "identity fp8", signed_zero=False)


def test_fp8_gemm_scale_fold_exact_and_deterministic():
    lib()
    codes, scale = synth.fp8_weight(512, 1024, seed=3)
    a = synth.bf16_activations(300, 1024, seed=4).to(DEV)
    w = codes.to(DEV)
    raw = gq.fp8_matmul(a, w, 1.0, out_dtype=torch.float32)
    s1 = gq.fp8_matmul(a, w, scale, out_dtype=torch.float32)
    s2 = gq.fp8_matmul(a, w, scale, out_dtype=torch.float32)
    assert torch.equal(s1, s2)
    assert torch.equal(s1, raw * torch.tensor(scale, dtype=torch.float32, device=DEV))


def test_fp8_gemm_row_equals_gemv():
    lib()
    codes, scale = synth.fp8_weight(640, 2048, seed=8)
    a = synth.bf16_activations(5, 2048, seed=9)
    c = to_f64(gq.fp8_matmul(a.to(DEV), codes.to(DEV), scale, out_dtype=torch.float32))
    w_hat = oracle.decode_fp8(codes.numpy())
    for i in range(5):
        y = to_f64(gq.fp8_gemv(a[i].to(DEV), codes.to(DEV), scale, out_dtype=torch.float32))
        tol = 2 * oracle.tolerance(bits(a)[i:i + 1], w_hat, scale)[0]
        assert_within(c[i], y, tol, f"gemm row {i} vs gemv")


def test_fp8_gemm_k_zero_writes_zeros():
    lib()
    a = torch.empty(3, 0, dtype=torch.bfloat16, device=DEV)
    w = torch.empty(5, 0, dtype=torch.uint8, device=DEV)
    c = torch.full((3, 5), 7.0, dtype=torch.float32, device=DEV)
    gq.fp8_matmul(a, w, 2.0, out=c)
    assert torch.all(c == 0)


def check_nvfp4(m, n, k, out_dtype=torch.float32, seed=0):
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=seed)
    a = synth.bf16_activations(m, k, seed=seed + 1)
    buf, c = canary_out((m, n), out_dtype)
    gq.nvfp4_matmul(a.to(DEV), q.to(DEV), bs.to(DEV), s2, out=c)
    torch.cuda.synchronize()
    assert_canary(buf)
    ab = bits(a)
    w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
    ref = oracle.linear(ab, w_hat, s2)
    tol = oracle.tolerance(ab, w_hat, s2, out_dtype == torch.bfloat16, ref=ref)
    assert_within(to_f64(c), ref, tol, f"nvfp4 gemm {m}x{n}x{k}")


@pytest.mark.parametrize("m", [1, 16, 128])
def test_nvfp4_gemm_config(m):
    lib()
    check_nvfp4(m, 4096, 4096, torch.bfloat16)


@pytest.mark.parametrize("m,n,k", [(3, 127, 64), (129, 300, 128), (200, 257, 576), (1, 1, 64)])
def test_nvfp4_gemm_shapes(m, n, k):
    lib()
    check_nvfp4(m, n, k, seed=m * 3 + n)


def test_nvfp4_gemm_identity_dequant_every_pair():
    """A = I recovers e2m1(q) * e4m3(bs) exactly for all code/scale pairs."""
    lib()
    k = 128
    n = 256
    rng = np.random.default_rng(1)
    q = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    bs = np.tile(np.arange(256, dtype=np.uint8)[:, None], (1, k // 16))
    bs = np.where(((bs & 0x7F) == 0x7F), 0x38, bs).astype(np.uint8)   # finite scales
    for j in range(k // 16):
        bs[:, j] = np.roll(bs[:, j], 17 * j)
    eye = torch.eye(k, dtype=torch.bfloat16)
    c = gq.nvfp4_matmul(eye.to(DEV), torch.from_numpy(q).to(DEV), torch.from_numpy(bs).to(DEV),
                        1.0, out_dtype=torch.float32)
    assert_exact(to_f64(c), oracle.nvfp4_materialize(q, bs).T, "identity nvfp4",
                 signed_zero=False)


def test_gemm_errors():
    l = lib()
    s = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(4, 32, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(8, 32, dtype=torch.uint8, device=DEV)
    c = torch.zeros(4, 8, dtype=torch.float32, device=DEV)
    assert l.gq_fp8_matmul(c.data_ptr(), 0, a.data_ptr(), w.data_ptr(), 4, 8, -1, 1.0, s) == 2
    assert l.gq_fp8_matmul(c.data_ptr(), 0, a.data_ptr() + 2, w.data_ptr(), 4, 8, 32, 1.0, s) == 3
    assert l.gq_fp8_matmul(c.data_ptr(), 0, None, w.data_ptr(), 4, 8, 32, 1.0, s) == 1
    assert l.gq_nvfp4_matmul(c.data_ptr(), 0, a.data_ptr(), w.data_ptr(), w.data_ptr(), 4, 8, 32,
                             1.0, s) == 2
    assert l.gq_fp8_matmul(c.data_ptr(), 0, a.data_ptr(), w.data_ptr(), 0, 8, 32, 1.0, s) == 0


def test_no_wait_timed_out():
    lib()
    torch.cuda.synchronize()
    assert gq.device_status() == 0


@pytest.mark.parametrize("m,n,k", [(16, 4096, 4096), (128, 1000, 4112), (100, 520, 2048),
                                   (128, 4096, 1024)])
def test_small_m_split_k(m, n, k):
    """M <= 128 with few N tiles: K is split over a thread-block cluster and
    the partials are reduced through distributed shared memory (uneven splits
    for K = 4112, N not a multiple of the tile)."""
    lib()
    check_fp8(m, n, k, seed=m + k)
    if k % 64 == 0:
        check_nvfp4(m, n, k, seed=m + k + 1)


def test_small_m_split_k_deterministic():
    lib()
    codes, s = synth.fp8_weight(4096, 4096, seed=50)
    a = synth.bf16_activations(64, 4096, seed=51).to(DEV)
    w = codes.to(DEV)
    r1 = gq.fp8_matmul(a, w, s, out_dtype=torch.float32)
    r2 = gq.fp8_matmul(a, w, s, out_dtype=torch.float32)
    assert torch.equal(r1, r2)


@pytest.mark.parametrize("m", [1, 2, 15, 16, 17, 31, 48, 64, 65, 100, 127, 128])
def test_small_m_every_row_count(m):
    """The few-row kernel (weight as the MMA's A operand, activations as B with
    N = M rounded up to 16): every padding case of M, N ragged (not a
    multiple of 4, so the scalar store path runs), bf16 and f32 outputs."""
    lib()
    check_fp8(m, 1003, 1024, torch.bfloat16 if m % 2 else torch.float32, seed=m)
    check_nvfp4(m, 1003, 1024, torch.float32 if m % 2 else torch.bfloat16, seed=m + 7)


@pytest.mark.parametrize("m,n,k", [(16, 14336, 4096), (128, 14336, 4096), (5, 4096, 14336)])
def test_small_m_decode_shapes(m, n, k):
    """Decode-batch shapes of the FP8 workload: many N tiles (no K split) and a
    long K with few tiles."""
    lib()
    check_fp8(m, n, k, torch.bfloat16, seed=m + n)


@pytest.mark.parametrize("m", [1, 40])
def test_small_m_short_k(m):
    """K of one or two stages (no split possible) and an FP8 K tail of 16."""
    lib()
    check_fp8(m, 384, 16, seed=3)
    check_fp8(m, 384, 80, seed=4)
    check_nvfp4(m, 384, 64, seed=5)
    check_nvfp4(m, 384, 128, seed=6)


def test_small_m_identity_dequant_every_fp8_code():
    """A = I with K = 128: the few-row kernel returns every E4M3 code's value
    (NaN codes poison their column)."""
    lib()
    k = 128
    codes = (np.arange(300 * k).reshape(300, k) * 11 % 256).astype(np.uint8)
    eye = torch.eye(k, dtype=torch.bfloat16)
    c = gq.fp8_matmul(eye.to(DEV), torch.from_numpy(codes).to(DEV), 1.0, out_dtype=torch.float32)
    want = oracle.fp8_materialize(codes).T.copy()
    nan_cols = np.isnan(oracle.fp8_materialize(codes)).any(axis=1)
    want[:, nan_cols] = np.nan
    assert_exact(to_f64(c), want, "identity fp8 (few rows)", signed_zero=False)


def test_small_m_nvfp4_unaligned_scales():
    """Block scales whose base is 4- but not 16-byte aligned cannot be loaded
    by TMA and take the general kernel; both placements match the oracle."""
    lib()
    q, bs, s2 = synth.nvfp4_weight(512, 4096, seed=21)
    a = synth.bf16_activations(16, 4096, seed=22)
    qd = q.to(DEV)
    store = torch.zeros(bs.numel() + 16, dtype=torch.uint8, device=DEV)
    shifted = store[4:4 + bs.numel()].view(bs.shape)
    shifted.copy_(bs.to(DEV))
    ab = bits(a)
    w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
    ref = oracle.linear(ab, w_hat, s2)
    tol = oracle.tolerance(ab, w_hat, s2, False, ref=ref)
    for scales in (bs.to(DEV), shifted):
        c = gq.nvfp4_matmul(a.to(DEV), qd, scales, s2, out_dtype=torch.float32)
        assert_within(to_f64(c), ref, tol, "nvfp4 scales placement")
