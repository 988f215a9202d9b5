"""Fused epilogue and binary16 output against the oracle.

    out = act(alpha * x @ dequant(W)^T + bias[n])     (grouped: bias[e, n])

through every product entry point's ``_ex`` form (both GEMM kernels: M <= 128
and M > 128), with each activation, f32 / bf16 / f16 bias and output types.
The tolerance is the matmul's (2e-4 |alpha| sum |x w|) carried through the
activation's Lipschitz bound, plus 2^-20 |out| for the fp32 bias add and
activation functions, plus one unit in the last place of the output type
(``oracle.tolerance_epilogue``).
"""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_canary, assert_exact, assert_within, bits, canary_out, lib, to_f64

pytestmark = pytest.mark.gpu

OUT_KIND = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}

# (activation, bias dtype or None, output dtype): each activation, each bias
# type and each output type appear.
CASES = [
    ("relu", torch.float32, torch.bfloat16),
    ("silu", torch.bfloat16, torch.float16),
    ("gelu_tanh", torch.float16, torch.float32),
    ("none", torch.float32, torch.float16),
    ("silu", None, torch.bfloat16),
]


def make_bias(shape, dtype, seed):
    if dtype is None:
        return None, None
    g = torch.Generator().manual_seed(seed)
    b = (torch.randn(shape, generator=g) * 0.5).to(dtype)
    return b.to(DEV), b.to(torch.float64).numpy()


def expected(pre, ab, w_hat, alpha, bias_f64, act, out_dtype):
    ref = oracle.epilogue(pre, bias_f64, act)
    tol_pre = oracle.tolerance(ab, w_hat, alpha)
    return ref, oracle.tolerance_epilogue(tol_pre, ref, act, OUT_KIND[out_dtype])


@pytest.mark.parametrize("act,bias_dtype,out_dtype", CASES)
@pytest.mark.parametrize("n,k", [(1000, 4096), (1003, 520), (2000, 4096)])
def test_fp8_gemv_epilogue(act, bias_dtype, out_dtype, n, k):
    lib()
    codes, scale = synth.fp8_weight(n, k, seed=n + k)
    x = synth.bf16_activations(1, k, seed=n + k + 1).reshape(-1)
    bias, bias64 = make_bias((n,), bias_dtype, n)
    buf, y = canary_out((n,), out_dtype)
    gq.fp8_gemv(x.to(DEV), codes.to(DEV), scale, out=y, bias=bias, activation=act)
    torch.cuda.synchronize()
    assert_canary(buf)
    ab = bits(x)[None, :]
    w_hat = oracle.decode_fp8(codes.numpy())
    ref, tol = expected(oracle.linear(ab, w_hat, scale), ab, w_hat, scale, bias64, act, out_dtype)
    assert_within(to_f64(y), ref[0], tol[0], f"fp8 gemv {act}")


@pytest.mark.parametrize("act,bias_dtype,out_dtype", CASES)
def test_nvfp4_gemv_epilogue(act, bias_dtype, out_dtype):
    lib()
    n, k = 1000, 4096
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=5)
    x = synth.bf16_activations(1, k, seed=6).reshape(-1)
    bias, bias64 = make_bias((n,), bias_dtype, 7)
    buf, y = canary_out((n,), out_dtype)
    gq.nvfp4_gemv(x.to(DEV), q.to(DEV), bs.to(DEV), s2, out=y, bias=bias, activation=act)
    torch.cuda.synchronize()
    assert_canary(buf)
    ab = bits(x)[None, :]
    w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
    ref, tol = expected(oracle.linear(ab, w_hat, s2), ab, w_hat, s2, bias64, act, out_dtype)
    assert_within(to_f64(y), ref[0], tol[0], f"nvfp4 gemv {act}")


@pytest.mark.parametrize("act,bias_dtype,out_dtype", CASES)
@pytest.mark.parametrize("m,n", [(16, 1000), (300, 1000), (40, 1003), (260, 1003)])
def test_fp8_matmul_epilogue(act, bias_dtype, out_dtype, m, n):
    """M <= 128 (few-row kernel) and M > 128; N = 1003 takes the scalar stores."""
    lib()
    k = 1024
    codes, scale = synth.fp8_weight(n, k, seed=m + n)
    a = synth.bf16_activations(m, k, seed=m + n + 1)
    bias, bias64 = make_bias((n,), bias_dtype, m)
    buf, c = canary_out((m, n), out_dtype)
    gq.fp8_matmul(a.to(DEV), codes.to(DEV), scale, out=c, bias=bias, activation=act)
    torch.cuda.synchronize()
    assert_canary(buf)
    ab = bits(a)
    w_hat = oracle.decode_fp8(codes.numpy())
    ref, tol = expected(oracle.linear(ab, w_hat, scale), ab, w_hat, scale, bias64, act, out_dtype)
    assert_within(to_f64(c), ref, tol, f"fp8 matmul {m}x{n} {act}")


@pytest.mark.parametrize("act,bias_dtype,out_dtype", CASES)
@pytest.mark.parametrize("m,n,k", [(16, 1000, 1024), (300, 1000, 1024), (100, 520, 192)])
def test_nvfp4_matmul_epilogue(act, bias_dtype, out_dtype, m, n, k):
    """M <= 128 with K % 256 == 0 (few-row kernel), M > 128, and M <= 128 with
    K % 256 != 0 (the general kernel's cluster split)."""
    lib()
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=m + 3)
    a = synth.bf16_activations(m, k, seed=m + 4)
    bias, bias64 = make_bias((n,), bias_dtype, m + 5)
    buf, c = canary_out((m, n), out_dtype)
    gq.nvfp4_matmul(a.to(DEV), q.to(DEV), bs.to(DEV), s2, out=c, bias=bias, activation=act)
    torch.cuda.synchronize()
    assert_canary(buf)
    ab = bits(a)
    w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
    ref, tol = expected(oracle.linear(ab, w_hat, s2), ab, w_hat, s2, bias64, act, out_dtype)
    assert_within(to_f64(c), ref, tol, f"nvfp4 matmul {m}x{n} {act}")


@pytest.mark.parametrize("act,bias_dtype,out_dtype", CASES)
def test_grouped_epilogue_bias_per_expert(act, bias_dtype, out_dtype):
    """Bias row of the group's expert; the -1 group stays zero (no epilogue);
    rows no group covers are untouched."""
    lib()
    e, n, k, total = 8, 320, 256, 600
    w, scales = synth.fp8_expert_stack(e, n, k, seed=9)
    a = synth.bf16_activations(total, k, seed=10)
    offs, ids, _ = synth.moe_routing(total - 40, seed=11)          # last 40 rows uncovered
    bias, bias64 = make_bias((e, n), bias_dtype, 12)
    c = torch.full((total, n), -7.25, dtype=out_dtype, device=DEV)
    gq.fp8_grouped_matmul(a.to(DEV), w.to(DEV), offs.to(torch.int32).to(DEV),
                          ids.to(torch.int32).to(DEV), scales.to(DEV), out=c, bias=bias,
                          activation=act)
    torch.cuda.synchronize()
    got = to_f64(c)
    ab = bits(a)
    offs_l, ids_l = offs.tolist(), ids.tolist()
    for z, ex in enumerate(ids_l):
        lo, hi = offs_l[z], offs_l[z + 1]
        if hi <= lo:
            continue
        if ex < 0:
            assert np.all(got[lo:hi] == 0.0), f"group {z} (-1) not zero"
            continue
        w_hat = oracle.decode_fp8(w[ex].numpy())
        s = float(scales[ex])
        b = None if bias64 is None else bias64[ex]
        ref, tol = expected(oracle.linear(ab[lo:hi], w_hat, s), ab[lo:hi], w_hat, s, b, act, out_dtype)
        assert_within(got[lo:hi], ref, tol, f"group {z} expert {ex} {act}")
    assert np.all(got[offs_l[-1]:] == -7.25)


def test_k_zero_gives_activation_of_bias():
    lib()
    a = torch.empty(3, 0, dtype=torch.bfloat16, device=DEV)
    w = torch.empty(5, 0, dtype=torch.uint8, device=DEV)
    bias = torch.tensor([-1.0, 0.0, 0.5, 2.0, -3.0], dtype=torch.float32, device=DEV)
    c = gq.fp8_matmul(a, w, 2.0, out_dtype=torch.float32, bias=bias, activation="silu")
    want = oracle.activation(bias.cpu().double().numpy(), "silu")
    tol = 2.0 ** -20 * np.abs(want) + 1e-30
    for r in range(3):
        assert_within(to_f64(c[r]), want, tol, "K = 0")


def test_epilogue_errors():
    l = lib()
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(32, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(8, 32, dtype=torch.uint8, device=DEV)
    y = torch.zeros(8, dtype=torch.float32, device=DEV)
    bias = torch.zeros(9, dtype=torch.float32, device=DEV)
    ep = gq.Epilogue(None, 0, 7)                                   # unknown activation
    assert l.gq_fp8_gemv_ex(y.data_ptr(), 0, x.data_ptr(), w.data_ptr(), 8, 32, 1.0,
                            gq._ref(ep), s) == 8
    ep = gq.Epilogue(bias.data_ptr(), 5, 0)                        # unknown bias dtype
    assert l.gq_fp8_gemv_ex(y.data_ptr(), 0, x.data_ptr(), w.data_ptr(), 8, 32, 1.0,
                            gq._ref(ep), s) == 8
    ep = gq.Epilogue(bias.data_ptr() + 2, 0, 0)                    # misaligned f32 bias
    assert l.gq_fp8_gemv_ex(y.data_ptr(), 0, x.data_ptr(), w.data_ptr(), 8, 32, 1.0,
                            gq._ref(ep), s) == 3
    assert l.gq_fp8_gemv(y.data_ptr(), 3, x.data_ptr(), w.data_ptr(), 8, 32, 1.0, s) == 4
    with pytest.raises(ValueError):
        gq.fp8_gemv(x, w, 1.0, bias=bias)                          # wrong bias shape
    with pytest.raises(ValueError):
        gq.fp8_gemv(x, w, 1.0, activation="tanh")


def test_grouped_k_zero_with_bias_is_rejected():
    lib()
    a = torch.empty(4, 0, dtype=torch.bfloat16, device=DEV)
    w = torch.empty(2, 8, 0, dtype=torch.uint8, device=DEV)
    offs = torch.tensor([0, 2, 4], dtype=torch.int32, device=DEV)
    ids = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    bias = torch.zeros(2, 8, dtype=torch.float32, device=DEV)
    with pytest.raises(gq.GQError):
        gq.fp8_grouped_matmul(a, w, offs, ids, bias=bias)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_materialize_f16_bit_exact(fmt):
    """Every decoded value is exact in binary16: the output bits equal the
    oracle's value rounded (exactly) to binary16."""
    lib()
    if fmt == "fp8":
        codes = (np.arange(256 * 48) % 256).astype(np.uint8).reshape(256, 48)
        o = gq.fp8_materialize(torch.from_numpy(codes).to(DEV), out_dtype=torch.float16)
        want = oracle.fp8_materialize(codes)
    else:
        q, bs, _ = synth.nvfp4_weight(64, 256, seed=3)
        bs = bs.clone()
        bs[0, :] = torch.arange(16, dtype=torch.uint8) * 7              # small and subnormal scales
        o = gq.nvfp4_materialize(q.to(DEV), bs.to(DEV), out_dtype=torch.float16)
        want = oracle.nvfp4_materialize(q.numpy(), bs.numpy())
    got_bits = o.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    finite = ~np.isnan(want)
    assert np.array_equal(got_bits[finite], oracle.f64_to_f16_bits(want)[finite])
    assert np.all(np.isnan(o.cpu().float().numpy()[~finite]))
    assert_exact(to_f64(o), want, f"{fmt} materialize f16")
