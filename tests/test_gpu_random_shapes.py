"""Seeded random shapes through every product entry point, against the oracle.

Each case draws its sizes, output type and epilogue from a fixed seed, so a
failure names a reproducible case.  Sizes stay small enough for the float64
oracle (a few hundred rows and columns) but cover ragged M, N and K (odd K
for the FP8 calls), the few-row and general GEMM kernels, and grouped calls
with empty, -1 and out-of-range groups; M up to 1100 reaches several CTA-pair
tiles.
"""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_within, bits, lib, to_f64

pytestmark = pytest.mark.gpu

OUT = [torch.float32, torch.bfloat16, torch.float16]
OUT_KIND = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
ACTS = ["none", "relu", "silu", "gelu_tanh"]


def _epi(rng, n, rows=None):
    """(bias tensor or None, bias float64 or None, activation)."""
    act = ACTS[rng.integers(0, len(ACTS))]
    if rng.random() < 0.5:
        shape = (n,) if rows is None else (rows, n)
        b = synth.gaussian(shape, 0.1, seed=int(rng.integers(1 << 30))).to(torch.bfloat16)
        return b, oracle.bf16_bits_to_f64(bits(b)), act
    return None, None, act


def _check(got, pre, tol_pre, bias64, act, out_dtype, what):
    ref = oracle.epilogue(pre, bias64, act)
    assert_within(got, ref, oracle.tolerance_epilogue(tol_pre, ref, act, OUT_KIND[out_dtype]), what)


@pytest.mark.parametrize("case", range(16))
def test_random_fp8_matmul(case):
    lib()
    rng = np.random.default_rng(1000 + case)
    m = int(rng.choice([1, 2, 7, 16, 64, 127, 128, 129, 300, 513, 700, 1100]))
    n = int(rng.integers(1, 700))
    k = int(rng.integers(1, 700)) if case % 2 else 16 * int(rng.integers(1, 40))
    out_dtype = OUT[case % 3]
    codes, s = synth.fp8_weight(n, k, seed=case)
    a = synth.bf16_activations(m, k, seed=case + 50)
    bias, b64, act = _epi(rng, n)
    c = gq.fp8_matmul(a.to(DEV), codes.to(DEV), s, out_dtype=out_dtype,
                      bias=None if bias is None else bias.to(DEV), activation=act)
    ab, w_hat = bits(a), oracle.decode_fp8(codes.numpy())
    _check(to_f64(c), oracle.linear(ab, w_hat, s), oracle.tolerance(ab, w_hat, s), b64, act,
           out_dtype, f"fp8_matmul {m}x{n}x{k} {out_dtype} {act}")


@pytest.mark.parametrize("case", range(12))
def test_random_nvfp4_matmul(case):
    lib()
    rng = np.random.default_rng(2000 + case)
    m = int(rng.choice([1, 5, 16, 100, 128, 129, 257, 513, 800]))
    n = int(rng.integers(1, 600))
    k = 64 * int(rng.integers(1, 16))
    out_dtype = OUT[case % 3]
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=case)
    a = synth.bf16_activations(m, k, seed=case + 60)
    bias, b64, act = _epi(rng, n)
    c = gq.nvfp4_matmul(a.to(DEV), q.to(DEV), bs.to(DEV), s2, out_dtype=out_dtype,
                        bias=None if bias is None else bias.to(DEV), activation=act)
    ab, w_hat = bits(a), oracle.decode_nvfp4(q.numpy(), bs.numpy())
    _check(to_f64(c), oracle.linear(ab, w_hat, s2), oracle.tolerance(ab, w_hat, s2), b64, act,
           out_dtype, f"nvfp4_matmul {m}x{n}x{k} {out_dtype} {act}")


@pytest.mark.parametrize("case", range(8))
def test_random_gemv(case):
    lib()
    rng = np.random.default_rng(3000 + case)
    n = int(rng.integers(1, 3000))
    out_dtype = OUT[case % 3]
    bias, b64, act = _epi(rng, n)
    if case % 2:
        k = int(rng.integers(1, 3000))
        codes, s = synth.fp8_weight(n, k, seed=case)
        x = synth.bf16_activations(1, k, seed=case + 70).reshape(-1)
        y = gq.fp8_gemv(x.to(DEV), codes.to(DEV), s, out_dtype=out_dtype,
                        bias=None if bias is None else bias.to(DEV), activation=act)
        xb, w_hat, alpha = bits(x)[None, :], oracle.decode_fp8(codes.numpy()), s
    else:
        k = 16 * int(rng.integers(1, 200))
        q, bs, s2 = synth.nvfp4_weight(n, k, seed=case)
        x = synth.bf16_activations(1, k, seed=case + 70).reshape(-1)
        y = gq.nvfp4_gemv(x.to(DEV), q.to(DEV), bs.to(DEV), s2, out_dtype=out_dtype,
                          bias=None if bias is None else bias.to(DEV), activation=act)
        xb, w_hat, alpha = bits(x)[None, :], oracle.decode_nvfp4(q.numpy(), bs.numpy()), s2
    _check(to_f64(y)[None, :], oracle.linear(xb, w_hat, alpha), oracle.tolerance(xb, w_hat, alpha),
           b64, act, out_dtype, f"gemv {n}x{k} {out_dtype} {act}")


@pytest.mark.parametrize("case", range(8))
def test_random_grouped(case):
    lib()
    rng = np.random.default_rng(4000 + case)
    e = int(rng.integers(1, 5))
    n = int(rng.integers(1, 500))
    k = 64 * int(rng.integers(1, 8))
    g = int(rng.integers(1, 7))
    sizes = rng.integers(0, 300, size=g)
    start = int(rng.integers(0, 5))
    offs = np.concatenate([[start], start + np.cumsum(sizes)]).astype(np.int64)
    total = int(offs[-1]) + int(rng.integers(0, 5))
    ids = rng.integers(-1, e + 1, size=g)          # includes -1 and one past the last expert
    a = synth.bf16_activations(max(total, 1), k, seed=case + 80)
    out_dtype = OUT[case % 3]
    bias, b64, act = _epi(rng, n, rows=e)
    out = torch.full((max(total, 1), n), -7.25, dtype=out_dtype, device=DEV)
    max_rows = int(max(sizes.max(), 1))
    kw = dict(max_rows_per_group=max_rows, out=out, bias=None if bias is None else bias.to(DEV),
              activation=act)
    d_offs = torch.as_tensor(offs, dtype=torch.int32).to(DEV)
    d_ids = torch.as_tensor(ids, dtype=torch.int32).to(DEV)
    ab = bits(a)
    if case % 2:
        stack, scales = synth.fp8_expert_stack(e, n, k, seed=case)
        gq.fp8_grouped_matmul(a.to(DEV), stack.to(DEV), d_offs, d_ids, scales.to(DEV), **kw)
        ref, written = oracle.fp8_grouped_matmul(ab, stack.numpy(), offs, ids, scales.numpy())
        decode = lambda j: oracle.decode_fp8(stack[j].numpy())
        sc = scales.numpy()
    else:
        q, bs, s2 = synth.nvfp4_expert_stack(e, n, k, seed=case)
        gq.nvfp4_grouped_matmul(a.to(DEV), q.to(DEV), bs.to(DEV), d_offs, d_ids, s2.to(DEV), **kw)
        ref, written = oracle.nvfp4_grouped_matmul(ab, q.numpy(), bs.numpy(), offs, ids, s2.numpy())
        decode = lambda j: oracle.decode_nvfp4(q[j].numpy(), bs[j].numpy())
        sc = s2.numpy()
    got = to_f64(out)
    assert np.all(got[~written[:got.shape[0]]] == -7.25)
    for z, ex in enumerate(ids):
        lo, hi = int(offs[z]), int(offs[z + 1])
        if hi <= lo:
            continue
        if ex < 0 or ex >= e:
            assert np.all(got[lo:hi] == 0.0), f"group {z} (id {ex}) not zero"
            continue
        w_hat = decode(int(ex))
        tol_pre = oracle.tolerance(ab[lo:hi], w_hat, float(sc[ex]))
        brow = None if b64 is None else b64[int(ex)]
        _check(got[lo:hi], ref[lo:hi], tol_pre, brow, act, out_dtype,
               f"grouped case {case} group {z}")


@pytest.mark.parametrize("case", range(6))
def test_random_w8a8(case):
    lib()
    rng = np.random.default_rng(5000 + case)
    if case < 4:
        m = int(rng.choice([1, 3, 16, 100, 128, 129, 300, 600]))
        n = int(rng.integers(1, 600))
        k = 16 * int(rng.integers(1, 40))
    else:   # long K: many float32 chunks added in int32 (small M: a split-K cluster)
        m = int(rng.choice([1, 3, 16, 100]))
        n = int(rng.integers(1, 200))
        k = 16 * int(rng.integers(1021, 2600))
    x = synth.bf16_activations(m, k, seed=case + 90)
    qa, sa = gq.int8_quantize_rows(x.to(DEV))
    want_q, want_s = oracle.int8_quantize_rows(bits(x))
    assert np.array_equal(qa.cpu().numpy(), want_q)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), want_s.view(np.uint32))
    qb, sb = synth.int8_weight(n, k, seed=case)
    out_dtype = OUT[case % 3]
    c = gq.int8_matmul(qa, qb.to(DEV), sa, sb.to(DEV), out_dtype=out_dtype)
    pre = oracle.int8_matmul(want_q, qb.numpy(), want_s, sb.numpy()).astype(np.float64)
    # the sums are exact int32, so only the output rounding separates the two
    _check(to_f64(c), pre, np.zeros_like(pre), None, "none", out_dtype, f"w8a8 {m}x{n}x{k}")
