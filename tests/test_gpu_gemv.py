"""GEMV kernels (M = 1 decode) against the oracle.

Tolerance (floating point): |gpu - oracle| <= 2e-4 * |alpha| * sum_k |x_k w_k|,
plus one bf16 ulp of the result for bf16 outputs (``oracle.tolerance``).
"""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import (DEV, assert_canary, assert_within, bits, canary_out, lib,
                            to_f64)

pytestmark = pytest.mark.gpu


def run_fp8(n, k, out_dtype, alpha_mode="scale", seed=0, x_offset=0, w_offset=0):
    codes, scale = synth.fp8_weight(n, k, seed=seed)
    x = synth.bf16_activations(1, k, seed=seed + 1).reshape(-1)
    alpha = scale if alpha_mode == "scale" else 1.0
    # optional misalignment: place the tensors at an element offset
    xs = torch.zeros(k + x_offset, dtype=torch.bfloat16, device=DEV)
    xs[x_offset:] = x.to(DEV)
    ws = torch.zeros(n * k + w_offset, dtype=torch.uint8, device=DEV)
    ws[w_offset:] = codes.reshape(-1).to(DEV)
    buf, y = canary_out((n,), out_dtype)
    gq.fp8_gemv(xs[x_offset:], ws[w_offset:].view(n, k), alpha, out=y)
    torch.cuda.synchronize()
    got = to_f64(y)
    w_hat = oracle.decode_fp8(codes.numpy())
    xb = bits(x)
    ref = oracle.fp8_gemv(xb, codes.numpy(), alpha)
    tol = oracle.tolerance(xb[None, :], w_hat, alpha, out_dtype == torch.bfloat16,
                           ref=ref[None, :])[0]
    assert_within(got, ref, tol, f"fp8 gemv {n}x{k}")
    assert_canary(buf)
    return got


# configs: N=256 K=512 / 520 fp32 (raw and scaled); decode shapes bf16 scaled
@pytest.mark.parametrize("k", [512, 520])
@pytest.mark.parametrize("alpha_mode", ["raw", "scale"])
def test_fp8_gemv_small_config(k, alpha_mode):
    lib()
    run_fp8(256, k, torch.float32, alpha_mode)


@pytest.mark.parametrize("n,k", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_fp8_gemv_decode_shapes(n, k):
    lib()
    run_fp8(n, k, torch.bfloat16)


@pytest.mark.parametrize("n", [1, 3, 127, 257])
@pytest.mark.parametrize("k", [0, 1, 16, 17, 32, 520, 4112])
def test_fp8_gemv_odd_shapes(n, k):
    lib()
    run_fp8(n, k, torch.float32, seed=n * 31 + k)


@pytest.mark.parametrize("x_offset,w_offset", [(1, 0), (0, 3), (2, 8), (4, 4)])
def test_fp8_gemv_misaligned_pointers(x_offset, w_offset):
    lib()
    run_fp8(65, 1024, torch.float32, x_offset=x_offset, w_offset=w_offset)


def test_fp8_gemv_scale_fold_is_exact_and_deterministic():
    """gemv(alpha) == fp32(gemv(1) * alpha) bit for bit, and repeat calls agree."""
    lib()
    codes, scale = synth.fp8_weight(1000, 4096, seed=5)
    x = synth.bf16_activations(1, 4096, seed=6).reshape(-1).to(DEV)
    w = codes.to(DEV)
    raw = gq.fp8_gemv(x, w, 1.0, out_dtype=torch.float32)
    scaled = gq.fp8_gemv(x, w, scale, out_dtype=torch.float32)
    again = gq.fp8_gemv(x, w, scale, out_dtype=torch.float32)
    assert torch.equal(scaled, again)
    assert torch.equal(scaled, raw * torch.tensor(scale, dtype=torch.float32, device=DEV))


def test_fp8_gemv_nan_code_propagates():
    lib()
    codes, _ = synth.fp8_weight(8, 256, seed=9)
    codes[3, 100] = 0x7F
    codes[5, 7] = 0xFF
    x = synth.bf16_activations(1, 256, seed=10).reshape(-1)
    got = gq.fp8_gemv(x.to(DEV), codes.to(DEV), 1.0, out_dtype=torch.float32).cpu().numpy()
    ref = oracle.layer.linear_loops(bits(x), oracle.decode_fp8(codes.numpy()), 1.0)[0]
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(got[3]) and np.isnan(got[5])


@pytest.mark.parametrize("case", ["large", "tiny", "inf", "nan", "exact"])
def test_fp8_gemv_activations_outside_binary16(case):
    """Activations far outside the binary16 range (beyond 65504, below its
    subnormal grid), infinities and NaNs: the oracle's result within the
    tolerance, and the IEEE specials where the definition has them."""
    lib()
    n, k = 1000, 4096
    codes, scale = synth.fp8_weight(n, k, seed=21)
    x = synth.bf16_activations(1, k, seed=22).reshape(-1).float()
    if case == "large":
        x[[5, 900, 4095]] = torch.tensor([1.0e6, -7.0e4, 3.0e5])
    elif case == "tiny":
        x[[0, 17, 2048]] = torch.tensor([3.0e-9, -1.0e-7, 2.5e-30])
    elif case == "inf":
        x[77] = float("inf")
    elif case == "nan":
        x[1234] = float("nan")
    x = x.to(torch.bfloat16)
    got = to_f64(gq.fp8_gemv(x.to(DEV), codes.to(DEV), scale, out_dtype=torch.float32))
    xb = bits(x)
    w_hat = oracle.decode_fp8(codes.numpy())
    ref = oracle.fp8_gemv(xb, codes.numpy(), scale)
    if case in ("inf", "nan"):
        assert np.array_equal(np.isnan(got), np.isnan(ref))
        fin = np.isfinite(ref)
        assert np.array_equal(got[~fin & ~np.isnan(ref)], ref[~fin & ~np.isnan(ref)])
        ref, got = ref[fin], got[fin]
        tol = oracle.tolerance(xb[None, :], w_hat, scale)[0][fin] if fin.any() else None
        if fin.any():
            assert_within(got, ref, tol, f"fp8 gemv {case}")
        return
    tol = oracle.tolerance(xb[None, :], w_hat, scale)[0]
    assert_within(got, ref, tol, f"fp8 gemv {case}")


def test_fp8_gemv_equals_gemm_row_of_oracle():
    """The GEMV of row i equals row i of the oracle's GEMM (within tolerance)."""
    lib()
    codes, scale = synth.fp8_weight(300, 2048, seed=12)
    a = synth.bf16_activations(3, 2048, seed=13)
    ref = oracle.fp8_matmul(bits(a), codes.numpy(), scale)
    w_hat = oracle.decode_fp8(codes.numpy())
    for i in range(3):
        got = to_f64(gq.fp8_gemv(a[i].to(DEV), codes.to(DEV), scale, out_dtype=torch.float32))
        tol = oracle.tolerance(bits(a)[i:i + 1], w_hat, scale)[0]
        assert_within(got, ref[i], tol, f"row {i}")


def run_nvfp4(n, k, out_dtype, seed=0):
    q, bs, s2 = synth.nvfp4_weight(n, k, seed=seed)
    x = synth.bf16_activations(1, k, seed=seed + 1).reshape(-1)
    buf, y = canary_out((n,), out_dtype)
    gq.nvfp4_gemv(x.to(DEV), q.to(DEV), bs.to(DEV), s2, out=y)
    torch.cuda.synchronize()
    got = to_f64(y)
    xb = bits(x)
    ref = oracle.nvfp4_gemv(xb, q.numpy(), bs.numpy(), s2)
    w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
    tol = oracle.tolerance(xb[None, :], w_hat, s2, out_dtype == torch.bfloat16, ref=ref[None, :])[0]
    assert_within(got, ref, tol, f"nvfp4 gemv {n}x{k}")
    assert_canary(buf)


def test_nvfp4_gemv_config():
    lib()
    run_nvfp4(4096, 4096, torch.bfloat16)


@pytest.mark.parametrize("n", [1, 3, 127, 257])
@pytest.mark.parametrize("k", [0, 16, 32, 48, 4112])
def test_nvfp4_gemv_odd_shapes(n, k):
    lib()
    run_nvfp4(n, k, torch.float32, seed=n + 7 * k)


def test_nvfp4_gemv_worked_example():
    """The hand-worked example of tests/golden/nvfp4_gemv_worked.txt."""
    lib()
    from tests import pins
    rows = pins._rows("nvfp4_gemv_worked.txt")
    q = torch.tensor([[int(c, 16) for c in rows["q"][0]]], dtype=torch.uint8, device=DEV)
    bs = torch.tensor([[int(c, 16) for c in rows["bs"][0]]], dtype=torch.uint8, device=DEV)
    x = torch.tensor([float(v) for v in rows["x"][0]], dtype=torch.bfloat16, device=DEV)
    y = gq.nvfp4_gemv(x, q, bs, float(rows["alpha"][0][0]), out_dtype=torch.float32)
    assert y.item() == float(rows["scaled"][0][0])


def test_gemv_errors():
    l = lib()
    s = torch.cuda.current_stream().cuda_stream
    w = torch.zeros(4, 32, dtype=torch.uint8, device=DEV)
    x = torch.zeros(32, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(4, dtype=torch.float32, device=DEV)
    assert l.gq_fp8_gemv(y.data_ptr(), 0, None, w.data_ptr(), 4, 32, 1.0, s) == 1
    assert l.gq_fp8_gemv(y.data_ptr(), 0, x.data_ptr(), w.data_ptr(), 4, -2, 1.0, s) == 2
    assert l.gq_fp8_gemv(y.data_ptr(), 5, x.data_ptr(), w.data_ptr(), 4, 32, 1.0, s) == 4
    assert l.gq_nvfp4_gemv(y.data_ptr(), 0, x.data_ptr(), w.data_ptr(), w.data_ptr(), 4, 24,
                           1.0, s) == 2
    assert l.gq_nvfp4_gemv(y.data_ptr(), 0, x.data_ptr() + 2, w.data_ptr(), w.data_ptr(), 4, 32,
                           1.0, s) == 3
    assert l.gq_fp8_gemv(y.data_ptr(), 0, x.data_ptr(), w.data_ptr(), 0, 32, 1.0, s) == 0


@pytest.mark.parametrize("n,k", [(1, 4096), (151, 4096), (152, 256), (153, 768), (5000, 2048),
                                 (7, 16384), (2, 32768)])
def test_gemv_row_splits(n, k):
    """Row counts below, at and above the SM count, ragged last CTA, long rows
    (the multi-vector unrolled loop plus its remainder) and short ones."""
    lib()
    run_fp8(n, k, torch.float32, seed=n)
    if k % 32 == 0:
        run_nvfp4(n, k, torch.float32, seed=n + 1)


@pytest.mark.parametrize("n,k", [(1216, 16), (1217, 4112), (2000, 16384), (1500, 12304),
                                 (3000, 8192), (3653, 1024), (20000, 256)])
def test_fp8_gemv_large_n(n, k):
    """Many rows per SM with 16-byte vectors: one vector per row (K = 16),
    threads with one to several vectors per row and a remainder past the
    unrolled batches (K = 4112, 12304), long rows (K = 16384) and a row count
    that leaves the last CTA ragged."""
    lib()
    run_fp8(n, k, torch.float32, seed=n + k)
    run_fp8(n, k, torch.bfloat16, seed=n + k + 1)


@pytest.fixture
def overlap_flag():
    """GQ_LAUNCH_OVERLAP_WEIGHT_READS on for the test, restored afterwards."""
    lib()
    old = gq.get_launch_flags()
    gq.set_launch_flags(gq.GQ_LAUNCH_OVERLAP_WEIGHT_READS)
    yield
    gq.set_launch_flags(old)


@pytest.mark.parametrize("n8", [1000, 3000])
def test_overlap_flag_gives_identical_results(overlap_flag, n8):
    codes, scale = synth.fp8_weight(n8, 4096, seed=21)
    q, bs, s2 = synth.nvfp4_weight(1000, 4096, seed=22)
    x = synth.bf16_activations(1, 4096, seed=23).reshape(-1).to(DEV)
    w, qd, bsd = codes.to(DEV), q.to(DEV), bs.to(DEV)
    on8 = gq.fp8_gemv(x, w, scale, out_dtype=torch.float32)
    on4 = gq.nvfp4_gemv(x, qd, bsd, s2, out_dtype=torch.float32)
    gq.set_launch_flags(0)
    off8 = gq.fp8_gemv(x, w, scale, out_dtype=torch.float32)
    off4 = gq.nvfp4_gemv(x, qd, bsd, s2, out_dtype=torch.float32)
    assert torch.equal(on8, off8) and torch.equal(on4, off4)


@pytest.mark.parametrize("n", [4096, 4104, 4098])
def test_overlap_flag_orders_activation_reads(overlap_flag, n):
    """A chain of dependent GEMVs (the output of one is the input of the next)
    and a torch kernel writing x right before a GEMV: with the overlap flag
    every x read still sees the previous kernel's result.  n = 4104 and 4098
    take the 8- and 2-byte weight-vector paths."""
    codes = [synth.fp8_weight(n, n, seed=30 + i)[0] for i in range(3)]
    ws = [c.to(DEV) for c in codes]
    x0 = synth.bf16_activations(1, n, seed=40).reshape(-1)
    xs = x0.to(DEV)
    outs = []
    for i in range(3):
        y = gq.fp8_gemv(xs, ws[i], 0.02, out_dtype=torch.bfloat16)
        outs.append(y)
        xs = y
    # torch writes x in place, then a GEMV reads it
    xt = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    xt.copy_(x0.to(DEV))
    yt = gq.fp8_gemv(xt, ws[0], 0.02, out_dtype=torch.float32)
    torch.cuda.synchronize()
    # reference chain on the oracle, each step from the GPU's bf16 input
    xin = bits(x0)
    for i in range(3):
        ref = oracle.fp8_gemv(xin, codes[i].numpy(), 0.02)
        tol = oracle.tolerance(xin[None, :], oracle.decode_fp8(codes[i].numpy()), 0.02, True,
                               ref=ref[None, :])[0]
        assert_within(to_f64(outs[i]), ref, tol, f"chain step {i}")
        xin = bits(outs[i].cpu())
    ref = oracle.fp8_gemv(bits(x0), codes[0].numpy(), 0.02)
    assert_within(to_f64(yt), ref, oracle.tolerance(bits(x0)[None, :],
                  oracle.decode_fp8(codes[0].numpy()), 0.02)[0], "after torch write")


@pytest.mark.parametrize("n,k", [(4096, 4096), (2048, 14336), (300, 1024)])
def test_plain_order_sees_weights_written_just_before(n, k):
    """Default launch flags: a torch kernel overwrites the weights right before
    the GEMV.  The GEMV prefetches its first weight bytes into L2 before it
    waits for that kernel; the values it reads must still be the new ones
    (whole-CTA prefetch at K = 4096 and 1024, row heads at K = 14336)."""
    lib()
    assert gq.get_launch_flags() == 0
    old8, scale = synth.fp8_weight(n, k, seed=70)
    new8, _ = synth.fp8_weight(n, k, seed=71)
    q_old, bs_old, s2 = synth.nvfp4_weight(n, k, seed=72)
    q_new, bs_new, _ = synth.nvfp4_weight(n, k, seed=73)
    x = synth.bf16_activations(1, k, seed=74).reshape(-1)
    xd = x.to(DEV)
    w = old8.to(DEV)
    q, bs = q_old.to(DEV), bs_old.to(DEV)
    new8_d, q_new_d, bs_new_d = new8.to(DEV), q_new.to(DEV), bs_new.to(DEV)
    gq.fp8_gemv(xd, w, scale, out_dtype=torch.float32)      # old weights once through L2
    gq.nvfp4_gemv(xd, q, bs, s2, out_dtype=torch.float32)
    w.copy_(new8_d)
    y8 = gq.fp8_gemv(xd, w, scale, out_dtype=torch.float32)
    q.copy_(q_new_d)
    bs.copy_(bs_new_d)
    y4 = gq.nvfp4_gemv(xd, q, bs, s2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    xb = bits(x)
    ref8 = oracle.fp8_gemv(xb, new8.numpy(), scale)
    assert_within(to_f64(y8), ref8,
                  oracle.tolerance(xb[None, :], oracle.decode_fp8(new8.numpy()), scale)[0],
                  "fp8 after weight write")
    ref4 = oracle.nvfp4_gemv(xb, q_new.numpy(), bs_new.numpy(), s2)
    assert_within(to_f64(y4), ref4,
                  oracle.tolerance(xb[None, :], oracle.decode_nvfp4(q_new.numpy(), bs_new.numpy()),
                                   s2)[0], "nvfp4 after weight write")


def test_launch_flags_reject_unknown_bits():
    lib()
    with pytest.raises(gq.GQError):
        gq.set_launch_flags(0x80)


def test_overlap_flag_orders_few_row_gemm(overlap_flag):
    """The few-row GEMM with the overlap flag: a chain of dependent products
    (each output, 16 x 512, is the next input) and a torch kernel writing
    the activations right before one; every activation read and output write
    stays ordered after the previous kernel."""
    m, n = 16, 512
    qs = [synth.nvfp4_weight(n, n, seed=50 + i) for i in range(3)]
    dq = [(q.to(DEV), bs.to(DEV)) for q, bs, _ in qs]
    a0 = synth.bf16_activations(m, n, seed=60)
    a = a0.to(DEV)
    outs = []
    for i in range(3):
        c = gq.nvfp4_matmul(a, dq[i][0], dq[i][1], qs[i][2], out_dtype=torch.bfloat16)
        outs.append(c)
        a = c
    at = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
    at.copy_(a0.to(DEV))
    ct = gq.nvfp4_matmul(at, dq[0][0], dq[0][1], qs[0][2], out_dtype=torch.float32)
    torch.cuda.synchronize()
    ain = bits(a0)
    for i in range(3):
        q, bs, s2 = qs[i]
        w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
        ref = oracle.nvfp4_matmul(ain, q.numpy(), bs.numpy(), s2)
        assert_within(to_f64(outs[i]), ref, oracle.tolerance(ain, w_hat, s2, True, ref=ref),
                      f"chain step {i}")
        ain = bits(outs[i].cpu())
    q, bs, s2 = qs[0]
    ref = oracle.nvfp4_matmul(bits(a0), q.numpy(), bs.numpy(), s2)
    assert_within(to_f64(ct), ref, oracle.tolerance(bits(a0), oracle.decode_nvfp4(q.numpy(), bs.numpy()), s2),
                  "after torch write")


def test_read_floor_probe():
    """gq_probe_gemv_read_floor runs both GEMV launch shapes with loads only:
    it returns GQ_OK, writes one checksum value per row (the number of the
    CTA's 128 threads whose folded words have the row's bit set: an integer in
    [0, 128]), and refuses bad arguments like the GEMVs."""
    lib()
    codes, _ = synth.fp8_weight(1000, 4096, seed=3)
    y = gq.probe_gemv_read_floor(codes.to(DEV))
    q, bs, _ = synth.nvfp4_weight(1000, 4096, seed=4)
    y4 = gq.probe_gemv_read_floor(q.to(DEV), bs.to(DEV))
    torch.cuda.synchronize()
    for v in (y, y4):
        vals = v.float().cpu()
        assert torch.all((vals >= 0) & (vals <= 128) & (vals == vals.round()))
    l = gq.load_library()
    s = torch.cuda.current_stream().cuda_stream
    w = codes.to(DEV)
    assert l.gq_probe_gemv_read_floor(2, y.data_ptr(), w.data_ptr(), None, 1000, 4096, s) == 4
    assert l.gq_probe_gemv_read_floor(0, y.data_ptr(), w.data_ptr(), None, 1000, 4100, s) == 2
    assert l.gq_probe_gemv_read_floor(1, y.data_ptr(), w.data_ptr(), None, 1000, 4096, s) == 1
    assert gq.device_status() == 0
