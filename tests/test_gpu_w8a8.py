"""W8A8 int8: the per-row activation quantizer and the int8 GEMM against the
oracle.

The quantizer takes its integer decisions in float32 like the oracle, so codes
and scales are compared bit for bit.  The GEMM's sum is the page's exact int32
accumulation for every input (the kernel sums chunks of at most 1024 K on
binary16 tensor-core products, each chunk exactly in float32, and adds the
chunks in int32), so the float32 dequant
((float32(acc) * a_scale) * b_scale, then bias) and the output rounding match
the oracle bit for bit, including sums far beyond 2^24.  Only an activation
adds tolerance: its float32 evaluation against the oracle's float64 one.
"""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_canary, assert_exact, assert_within, bits, canary_out, lib, to_f64

pytestmark = pytest.mark.gpu


def out_bits_f64(v32, out_dtype):
    """Oracle float32 values -> the values of the output type, rounded RNE."""
    v = np.asarray(v32, dtype=np.float64)
    if out_dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(v))
    if out_dtype == torch.float16:
        return oracle.f16_bits_to_f64(oracle.f64_to_f16_bits(v))
    return v


def check_quantize(m, k, seed, special=False):
    x = synth.bf16_activations(m, k, seed=seed)
    if special and m >= 3:
        x[0] = 0
        row = torch.zeros(k)
        row[0] = 127
        vals = torch.tensor([2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.5])
        row[1:1 + min(7, k - 1)] = vals[:min(7, k - 1)]
        x[1] = row.to(torch.bfloat16)
    q, s = gq.int8_quantize_rows(x.to(DEV))
    torch.cuda.synchronize()
    want_q, want_s = oracle.int8_quantize_rows(bits(x))
    assert np.array_equal(q.cpu().numpy(), want_q), "codes differ"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), want_s.view(np.uint32)), "scales differ"


@pytest.mark.parametrize("m,k", [(1, 16), (3, 64), (257, 4096), (64, 8192), (5, 8208),
                                 (7, 100), (33, 5), (2, 1), (2048, 4096)])
def test_quantize_rows_exact(m, k):
    """Codes and scales bit for bit (rows with exact ties to even, zero
    rows, K with and without the register kernel)."""
    lib()
    check_quantize(m, k, seed=m + k, special=True)


def quantize_domain_rows():
    """One row per positive bf16 absmax a whose scale a / 127 is a normal
    float32: a itself, then every bf16 magnitude in [a / 256, a] (1025
    patterns, or down to zero) with both signs, zero-padded to K = 2064.
    Every quotient x / scale with |code| >= 1 that the quantizer can meet
    is in there."""
    top = np.arange(0x0080, 0x7F80, dtype=np.int32)            # positive normal bf16
    a = (top.astype(np.uint32) << 16).view(np.float32)
    top = top[(a / np.float32(127.0)) >= np.float32(2.0 ** -126)]
    k = 2064
    rows = np.zeros((top.size, k), dtype=np.uint16)
    mags = np.maximum(top[:, None] - np.arange(0, 1025, dtype=np.int32)[None, :], 0)
    rows[:, 0] = top
    rows[:, 1:1026] = mags
    rows[:, 1026:2051] = mags | 0x8000
    return torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16)


def test_quantize_exhaustive_quotients():
    """The register kernel divides by the row's scale with Markstein's
    correction step (one reciprocal per row, a product, a fused residual and
    a fused correction): its codes must equal the IEEE float32 division's on
    every quotient it can meet.  Codes and scales bit for bit against the
    oracle for every normal scale and every bf16 activation from absmax / 256
    to absmax, both signs (31 K rows, 65 M quotients)."""
    lib()
    x = quantize_domain_rows()
    q, s = gq.int8_quantize_rows(x.to(DEV))
    torch.cuda.synchronize()
    want_q, want_s = oracle.int8_quantize_rows(bits(x))
    got_q = q.cpu().numpy()
    bad = np.argwhere(got_q != want_q)
    assert bad.size == 0, f"{len(bad)} codes differ, first at row, col {bad[:3].tolist()}"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), want_s.view(np.uint32)), "scales differ"


def test_quantize_rows_unaligned_rows():
    """A row pitch that is not a multiple of 16 bytes takes the element-wise
    kernel; a view starting 2 bytes in does too."""
    lib()
    x = synth.bf16_activations(9, 72, seed=3).to(DEV)
    q, s = gq.int8_quantize_rows(x)
    want_q, want_s = oracle.int8_quantize_rows(bits(x.cpu()))
    assert np.array_equal(q.cpu().numpy(), want_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), want_s.view(np.uint32))


def run_matmul(qa, sa, qb, sb, out_dtype=torch.bfloat16, bias=None, act="none", rows=None):
    m, n = qa.shape[0], qb.shape[0]
    buf, c = canary_out((m, n), out_dtype)
    gq.int8_matmul(qa.to(DEV), qb.to(DEV), sa.to(DEV), sb.to(DEV), out=c,
                   bias=None if bias is None else bias.to(DEV), activation=act)
    torch.cuda.synchronize()
    assert_canary(buf)
    got = to_f64(c)
    sel = np.arange(m) if rows is None else np.asarray(rows)
    qa_s, sa_s = qa.numpy()[sel], sa.numpy()[sel]
    b64 = None if bias is None else oracle.bf16_bits_to_f64(bits(bias))
    pre = oracle.int8_matmul(qa_s, qb.numpy(), sa_s, sb.numpy(), b64)
    if act == "none":
        assert_exact(got[sel], out_bits_f64(pre, out_dtype), f"int8 {m}x{n}x{qa.shape[1]}")
        return got
    # The pre-activation value is the oracle's float32 bit for bit; the
    # activation is evaluated in float32 on the GPU and in float64 here: a few
    # float32 ulps of its input (2^-22 |pre|) and of its output.
    ref = oracle.epilogue(pre.astype(np.float64), None, act)
    out_kind = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[out_dtype]
    tol = oracle.tolerance_epilogue(2.0 ** -22 * np.abs(pre), ref, act, out_kind)
    assert_within(got[sel], ref, tol, f"int8 {m}x{n}x{qa.shape[1]} {act}")
    return got


@pytest.mark.parametrize("m,n,k", [(1, 256, 16), (16, 4096, 4096), (128, 384, 256), (129, 257, 64),
                                   (300, 1000, 2048), (512, 512, 1024), (3, 7, 32), (260, 96, 1040)])
def test_int8_matmul_exact(m, n, k):
    lib()
    qa, sa = synth.int8_codes(m, k, seed=m + k)
    qb, sb = synth.int8_weight(n, k, seed=n + k)
    run_matmul(qa, sa, qb, sb)


@pytest.mark.parametrize("m,n,k", [(129, 129, 64), (256, 200, 128), (257, 300, 256), (700, 520, 192)])
def test_int8_matmul_pair_tile_edges(m, n, k):
    """M > 128 runs on CTA pairs: tiles of 256 rows (128 per CTA) and 256
    weight rows (128 per CTA); row counts around the tile edges, N with the
    odd CTA's weight rows partly or wholly past the end."""
    lib()
    qa, sa = synth.int8_codes(m, k, seed=2 * m + k)
    qb, sb = synth.int8_weight(n, k, seed=3 * n + k)
    run_matmul(qa, sa, qb, sb)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_int8_matmul_out_types(out_dtype):
    lib()
    qa, sa = synth.int8_codes(200, 512, seed=1)
    qb, sb = synth.int8_weight(320, 512, seed=2)
    run_matmul(qa, sa, qb, sb, out_dtype)


def test_int8_matmul_bias_exact_and_activations():
    lib()
    qa, sa = synth.int8_codes(140, 256, seed=4)
    qb, sb = synth.int8_weight(272, 256, seed=5)
    bias = synth.gaussian((272,), 0.1, seed=6).to(torch.bfloat16)
    run_matmul(qa, sa, qb, sb, bias=bias)
    for act in ("relu", "silu", "gelu_tanh"):
        run_matmul(qa, sa, qb, sb, bias=bias, act=act)


def test_int8_large_sums_exact():
    """Uniform codes with K = 8192: sums of |a b| reach 2^25, beyond what a
    float32 accumulator holds exactly; the result is still the exact int32
    sum (bit-exact output)."""
    lib()
    qa, sa = synth.int8_codes(130, 8192, seed=7)
    qb, _ = synth.int8_codes(256, 8192, seed=8)
    sb = torch.full((256,), 0.01, dtype=torch.float32)
    run_matmul(qa, sa, qb, sb, out_dtype=torch.float32)


def extreme_codes(m, k, seed):
    """Codes drawn from {-128, -127, 127} (the extremes of int8 and of the
    quantizer's range) with rows of one sign, so that the sums reach
    128 * 128 * K and every partial sum of a float32 accumulator in natural
    order leaves the exact range early."""
    g = torch.Generator().manual_seed(seed)
    pick = torch.tensor([-128, -127, 127], dtype=torch.int16)
    codes = pick[torch.randint(0, 3, (m, k), generator=g)]
    codes[0] = 127
    codes[1] = -128
    if m > 2:
        codes[2] = -127
    return codes.to(torch.int8)


@pytest.mark.parametrize("m,n,k", [(130, 256, 4096), (5, 300, 16320), (3, 64, 16384),
                                   (129, 260, 24576), (2, 40, 65536), (3, 8, 130560),
                                   (257, 256, 1024), (300, 256, 1040), (129, 128, 2048),
                                   (4, 64, 1024), (6, 48, 3072), (260, 16, 130560)])
def test_int8_extreme_codes_exact(m, n, k):
    """All codes at +-127 / -128 (every chunk of 1024 K reaches the float32
    exact limit 2^24), K from one chunk (1024) and a chunk plus one 16-K step
    (1040) through 4096 (127^2 * 4096 ~ 2^26) up to 130560 (sums near 2^31),
    on CTA pairs (M > 128) and on one-CTA tiles with and without a split-K
    cluster: bit-exact against the exact int32 sums of the oracle."""
    lib()
    qa = extreme_codes(m, k, seed=m + k)
    qb = extreme_codes(n, k, seed=n + 3 * k)
    sa = torch.full((m,), 1.0, dtype=torch.float32)
    sb = (torch.rand(n, generator=torch.Generator().manual_seed(k)) + 0.5).to(torch.float32)
    got = run_matmul(qa, sa, qb, sb, out_dtype=torch.float32)
    # row 0 (all 127) against row 1 of the weight (all -128): -127 * 128 * K,
    # far beyond 2^24
    assert got[0, 1] == np.float32(np.float32(-127 * 128 * k) * np.float32(sb[1].item()))


def test_int8_k_limit():
    """K beyond 130560 (where |acc| could leave int32) is refused with
    GQ_ERR_TOO_LARGE before anything is queued."""
    lib()
    l = gq.load_library()
    s = torch.cuda.current_stream().cuda_stream
    k = 130560 + 16
    a = torch.zeros((2, k), dtype=torch.int8, device=DEV)
    c = torch.zeros((2, 8), dtype=torch.float32, device=DEV)
    sc = torch.ones(8, device=DEV)
    assert l.gq_int8_matmul(c.data_ptr(), 0, a.data_ptr(), a.data_ptr(), sc.data_ptr(),
                            sc.data_ptr(), 2, 8, k, s) == 7


def test_w8a8_pipeline_prefill_sampled():
    """x [2048, 4096] bf16 -> quantize (bit-exact) -> int8 GEMM with the
    [14336, 4096] int8 weight, bf16 out, checked on sampled rows."""
    lib()
    x = synth.bf16_activations(2048, 4096, seed=1)
    qb, sb = synth.int8_weight(14336, 4096, seed=0)
    qa_d, sa_d = gq.int8_quantize_rows(x.to(DEV))
    qa, sa = oracle.int8_quantize_rows(bits(x))
    assert np.array_equal(qa_d.cpu().numpy(), qa)
    assert np.array_equal(sa_d.cpu().numpy().view(np.uint32), sa.view(np.uint32))
    rng = np.random.default_rng(3)
    rows = sorted(set([0, 1, 127, 128, 255, 2047] + list(rng.integers(0, 2048, 20))))
    run_matmul(torch.from_numpy(qa), torch.from_numpy(sa), qb, sb, rows=rows)


def test_int8_k_zero_and_errors():
    lib()
    l = gq.load_library()
    s = torch.cuda.current_stream().cuda_stream
    qa = torch.zeros((4, 0), dtype=torch.int8, device=DEV)
    qb = torch.zeros((8, 0), dtype=torch.int8, device=DEV)
    sa = torch.ones(4, device=DEV)
    sb = torch.ones(8, device=DEV)
    bias = torch.arange(8, dtype=torch.float32, device=DEV)
    c = gq.int8_matmul(qa, qb, sa, sb, out_dtype=torch.float32, bias=bias)
    assert torch.equal(c.cpu(), bias.cpu().expand(4, 8))
    a = torch.zeros((4, 24), dtype=torch.int8, device=DEV)
    c = torch.zeros((4, 8), dtype=torch.float32, device=DEV)
    assert l.gq_int8_matmul(c.data_ptr(), 0, a.data_ptr(), a.data_ptr(), sa.data_ptr(),
                            sb.data_ptr(), 4, 8, 24, s) == 2
    assert l.gq_int8_matmul(c.data_ptr(), 0, a.data_ptr(), a.data_ptr(), None, sb.data_ptr(),
                            4, 8, 16, s) == 1


def test_quantize_exact_ties_and_tiny_rows():
    """Rows whose quotients are exact half-integers (scale a power of two),
    rows of tiny magnitude (the scale far below normal activations, down to
    bf16 subnormals), and random rows: codes and scales bit-exact."""
    lib()
    k = 256
    g = torch.Generator().manual_seed(9)
    rows = []
    for e in (-3, 0, 4):
        s = 2.0 ** e
        r = (torch.randint(-127, 127, (k,), generator=g).to(torch.float32) + 0.5) * s
        r[0] = 127 * s
        rows.append(r)
    for e in (-100, -125, -133):
        rows.append(torch.randn(k, generator=g) * 2.0 ** e)
    rows.append(torch.randn(k, generator=g) * 1e3)
    x = torch.stack(rows).to(torch.bfloat16)
    q, s = gq.int8_quantize_rows(x.to(DEV))
    want_q, want_s = oracle.int8_quantize_rows(bits(x))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), want_s.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), want_q)


def test_quantize_rows_k_zero_and_m_zero():
    lib()
    x = torch.zeros((3, 0), dtype=torch.bfloat16, device=DEV)
    q, s = gq.int8_quantize_rows(x)
    assert q.shape == (3, 0) and torch.equal(s.cpu(), torch.zeros(3))
    x = torch.zeros((0, 32), dtype=torch.bfloat16, device=DEV)
    q, s = gq.int8_quantize_rows(x)
    assert q.shape == (0, 32) and s.numel() == 0
