"""FP8 GEMM with K not a multiple of 16: the residue-class staging path.

Rows of A (2K bytes) and W (K bytes) are then not 16-byte strided: rows 8
(A) and 16 (W) apart are, so one TMA box per residue class brings the
16-byte-aligned windows that are realigned in shared memory (A by a plain
tiled box when K % 8 == 0); the K tail of the last stage is zero.  Same tolerance as the aligned GEMM:
|gpu - oracle| <= 2e-4 * |alpha| * sum_k |a_k w_k| (+1 ulp of the output type).
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


def exact_tensor(t):
    """A device copy in an allocation of exactly its own size, so that a read
    past the last byte of A or W would leave the buffer."""
    out = torch.empty(t.numel(), dtype=t.dtype, device=DEV)
    out.copy_(t.reshape(-1))
    return out.view(t.shape)


def check(m, n, k, out_dtype=torch.float32, seed=0, rows=None, bias=None, act="none"):
    codes, scale = synth.fp8_weight(n, k, seed=seed)
    a = synth.bf16_activations(m, k, seed=seed + 1)
    buf, c = canary_out((m, n), out_dtype)
    gq.fp8_matmul(exact_tensor(a), exact_tensor(codes), scale, out=c,
                  bias=None if bias is None else bias.to(DEV), activation=act)
    torch.cuda.synchronize()
    assert_canary(buf)
    got = to_f64(c)
    sel = np.arange(m) if rows is None else np.asarray(rows)
    ab = bits(a)[sel]
    w_hat = oracle.decode_fp8(codes.numpy())
    pre = oracle.linear(ab, w_hat, scale)
    out_kind = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[out_dtype]
    ref = oracle.epilogue(pre, None if bias is None else oracle.bf16_bits_to_f64(bits(bias)), act)
    tol = oracle.tolerance_epilogue(oracle.tolerance(ab, w_hat, scale), ref, act, out_kind)
    assert_within(got[sel], ref, tol, f"fp8 gemm any-K {m}x{n}x{k}")
    return c


@pytest.mark.parametrize("m,n,k", [(1, 256, 1), (3, 5, 7), (17, 33, 3), (200, 384, 520),
                                   (130, 257, 65), (257, 300, 129), (513, 700, 1001),
                                   (64, 4096, 4099), (300, 1000, 4100), (129, 520, 2),
                                   (513, 700, 1000), (7, 40, 8), (260, 300, 24), (128, 256, 4104),
                                   (5, 33, 4102), (100, 67, 12)])
def test_anyk_shapes(m, n, k):
    lib()
    check(m, n, k, seed=m + n + k)


# M > 256 runs on CTA pairs: each CTA realigns 256 rows of A (tile rows
# 256 rank + [0, 256)) and decodes 128 weight rows.  Rows just past 256 and
# 512, N below 16 (no weight box at all) or with the odd CTA's weight rows
# partly or wholly past the end, K with and without the plain A box, and
# every W residue count R = 16 / gcd(K, 16) (2, 4, 8, 16) with N % R rows
# past the last full group, and every A class count 8 / gcd(K, 8) (2, 4, 8)
# with M % R_A rows past the last full group.
@pytest.mark.parametrize("m,n,k", [(257, 129, 72), (511, 129, 100), (600, 200, 100), (777, 15, 33),
                                   (1030, 130, 4104), (513, 260, 4100), (700, 259, 4102),
                                   (600, 131, 1004), (300, 1001, 4100), (515, 64, 70),
                                   (701, 40, 4102)])
def test_anyk_pair_edges(m, n, k):
    lib()
    check(m, n, k, seed=2 * m + n + k)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_anyk_out_types(out_dtype):
    lib()
    check(300, 512, 777, out_dtype, seed=4)


def test_anyk_epilogue():
    lib()
    bias = synth.gaussian((448,), 0.05, seed=9).to(torch.bfloat16)
    check(260, 448, 333, torch.bfloat16, seed=8, bias=bias, act="silu")


@pytest.mark.parametrize("k", [4100, 4104])
def test_anyk_prefill_sampled(k):
    """M=2048, N=14336 with K=4100 and 4104 (the prefill shape with a ragged
    K; 4104 takes the plain A box); the oracle checks sampled rows."""
    lib()
    rng = np.random.default_rng(1)
    rows = sorted(set([0, 1, 127, 128, 255, 2047] + list(rng.integers(0, 2048, 30))))
    check(2048, 14336, k, torch.bfloat16, seed=3, rows=rows)


def test_anyk_identity_every_code():
    """A = I (K = 250 rows): the product returns every decoded code exactly,
    including subnormals and -0 (as +0: the result is 1 * w + 0 * others).  A
    column of W holding a NaN code is NaN in every row (0 * NaN = NaN)."""
    lib()
    k = 250
    n = 300
    codes = (np.arange(n * k).reshape(n, k) * 7 % 256).astype(np.uint8)
    eye = torch.eye(k, dtype=torch.bfloat16)
    c = gq.fp8_matmul(exact_tensor(eye), exact_tensor(torch.from_numpy(codes)), 1.0,
                      out_dtype=torch.float32)
    w_hat = oracle.decode_fp8(codes)
    want = w_hat.T.copy()
    want[:, np.isnan(w_hat).any(axis=1)] = np.nan
    assert_exact(to_f64(c), want, "identity any-K", signed_zero=False)


def test_anyk_deterministic_and_matches_gemv_row():
    lib()
    m, n, k = 150, 640, 1003
    codes, scale = synth.fp8_weight(n, k, seed=12)
    a = synth.bf16_activations(m, k, seed=13)
    da, dw = a.to(DEV), codes.to(DEV)
    c1 = gq.fp8_matmul(da, dw, scale, out_dtype=torch.float32)
    c2 = gq.fp8_matmul(da, dw, scale, out_dtype=torch.float32)
    assert torch.equal(c1.view(torch.int32), c2.view(torch.int32))
    y = gq.fp8_gemv(da[77].contiguous(), dw, scale, out_dtype=torch.float32)
    ab = bits(a)[77:78]
    tol = 2 * oracle.tolerance(ab, oracle.decode_fp8(codes.numpy()), scale)[0]
    assert_within(to_f64(c1)[77], to_f64(y), tol, "row 77 vs gemv")


def test_anyk_k_limit():
    """K not a multiple of 16 is limited to 2^27 (tensor-map coordinates);
    the call is refused before any launch."""
    l = lib()
    s = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(16, dtype=torch.uint8, device=DEV)
    c = torch.zeros(4, dtype=torch.float32, device=DEV)
    assert l.gq_fp8_matmul(c.data_ptr(), 0, a.data_ptr(), w.data_ptr(), 1, 1, (1 << 27) + 1,
                           1.0, s) == 7
