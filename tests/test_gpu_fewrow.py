"""Products with at most 16 activation rows (the register-fed mma.sync path
of fewrow.cu) against the oracle: every row count 1..16, ragged N, several K
(the FP8 path needs K % 64 == 0, NVFP4 K % 128 == 0; other K take the
tcgen05 few-row kernel), the fused epilogue and all output types, sampled
rows at the config shape, determinism, and an output canary."""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_canary, assert_within, bits, canary_out, lib, to_f64

pytestmark = pytest.mark.gpu

OUT_KIND = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


def run(fmt, m, n, k, out_dtype=torch.float32, seed=0, bias=False, act="none"):
    a = synth.bf16_activations(m, k, seed=seed + 1)
    ab = bits(a)
    b = synth.gaussian((n,), 0.05, seed=seed + 2).to(torch.bfloat16) if bias else None
    buf, c = canary_out((m, n), out_dtype)
    kw = dict(out=c, bias=None if b is None else b.to(DEV), activation=act)
    if fmt == "fp8":
        codes, s = synth.fp8_weight(n, k, seed=seed)
        w_hat = oracle.decode_fp8(codes.numpy())
        gq.fp8_matmul(a.to(DEV), codes.to(DEV), s, **kw)
    else:
        q, bs, s = synth.nvfp4_weight(n, k, seed=seed)
        w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
        gq.nvfp4_matmul(a.to(DEV), q.to(DEV), bs.to(DEV), s, **kw)
    torch.cuda.synchronize()
    assert_canary(buf)
    pre = oracle.linear(ab, w_hat, s)
    tol = oracle.tolerance(ab, w_hat, s)
    b64 = None if b is None else oracle.bf16_bits_to_f64(synth.bf16_bits(b))
    ref = oracle.epilogue(pre, b64, act)
    tol = oracle.tolerance_epilogue(tol, ref, act, OUT_KIND[out_dtype])
    assert_within(to_f64(c), ref, tol, f"{fmt} few-row {m}x{n}x{k} {act}")
    return c


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("m", list(range(1, 17)))
def test_every_row_count(fmt, m):
    run(fmt, m, 272, 256, seed=m)


@pytest.mark.parametrize("fmt,n,k", [("fp8", 1, 64), ("fp8", 17, 128), ("fp8", 1000, 4096),
                                     ("fp8", 333, 8192), ("nvfp4", 1, 128), ("nvfp4", 15, 256),
                                     ("nvfp4", 1000, 4096), ("nvfp4", 300, 14336),
                                     ("nvfp4", 37, 384), ("nvfp4", 9, 640)])
def test_shapes(fmt, n, k):
    lib()
    for m in (3, 9, 16):
        run(fmt, m, n, k, seed=n + k + m)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("act", ["relu", "silu", "gelu_tanh"])
def test_epilogue_and_output_types(out_dtype, act):
    lib()
    run("nvfp4", 12, 200, 512, out_dtype, seed=5, bias=True, act=act)
    run("fp8", 7, 200, 512, out_dtype, seed=6, bias=True, act=act)


def test_config_shape_nvfp4_m16():
    """The NVFP4 config: M = 16, N = K = 4096, bf16 out, every output."""
    lib()
    run("nvfp4", 16, 4096, 4096, torch.bfloat16, seed=0)


def test_deterministic():
    lib()
    q, bs, s = synth.nvfp4_weight(512, 2048, seed=8)
    a = synth.bf16_activations(16, 2048, seed=9).to(DEV)
    r1 = gq.nvfp4_matmul(a, q.to(DEV), bs.to(DEV), s, out_dtype=torch.float32)
    r2 = gq.nvfp4_matmul(a, q.to(DEV), bs.to(DEV), s, out_dtype=torch.float32)
    assert torch.equal(r1, r2)
    assert gq.device_status() == 0


def test_nan_code_propagates():
    """An E4M3 NaN code in one weight row makes exactly that output column NaN."""
    lib()
    codes, s = synth.fp8_weight(64, 256, seed=10)
    codes[5, 17] = 0x7F
    a = synth.bf16_activations(4, 256, seed=11)
    c = gq.fp8_matmul(a.to(DEV), codes.to(DEV), s, out_dtype=torch.float32).cpu()
    assert torch.isnan(c[:, 5]).all()
    assert not torch.isnan(c[:, :5]).any() and not torch.isnan(c[:, 6:]).any()
