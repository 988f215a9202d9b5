"""Grouped (MoE) NVFP4 GEMM against the oracle's per-group definition."""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_exact, assert_within, bits, lib, to_f64

pytestmark = pytest.mark.gpu

SENTINEL = -7.25


def run_grouped(a, q, bs, scales, offs, ids, max_rows, out_dtype=torch.float32, rows=None,
                bias=None, activation="none"):
    total_m = a.shape[0]
    n = q.shape[1]
    out = torch.full((total_m, n), SENTINEL, dtype=out_dtype, device=DEV)
    gq.nvfp4_grouped_matmul(a.to(DEV), q.to(DEV), bs.to(DEV),
                            torch.as_tensor(offs, dtype=torch.int32).to(DEV),
                            torch.as_tensor(ids, dtype=torch.int32).to(DEV),
                            None if scales is None else scales.to(DEV),
                            max_rows_per_group=max_rows, out=out,
                            bias=None if bias is None else bias.to(DEV), activation=activation)
    torch.cuda.synchronize()
    got = to_f64(out)
    ab = bits(a)
    ref, written = oracle.nvfp4_grouped_matmul(ab, q.numpy(), bs.numpy(), np.asarray(offs),
                                               np.asarray(ids),
                                               None if scales is None else scales.numpy(),
                                               rows=rows)
    assert np.all(got[~written] == SENTINEL)
    offs = np.asarray(offs)
    out_kind = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[out_dtype]
    for z, e in enumerate(np.asarray(ids)):
        r0, r1 = int(offs[z]), int(offs[z + 1])
        if r1 <= r0:
            continue
        sel = np.arange(r0, r1) if rows is None else np.intersect1d(np.arange(r0, r1), rows)
        if sel.size == 0:
            continue
        if e < 0 or e >= q.shape[0]:
            assert np.all(got[sel] == 0.0), f"group {z} (id {e}) must be zero"
            continue
        w_hat = oracle.decode_nvfp4(q[e].numpy(), bs[e].numpy())
        s = 1.0 if scales is None else float(scales[e])
        tol_pre = oracle.tolerance(ab[sel], w_hat, s)
        want = ref[sel]
        if bias is not None or activation != "none":
            b = None if bias is None else oracle.bf16_bits_to_f64(bits(bias[e]))
            want = oracle.epilogue(want, b, activation)
        tol = oracle.tolerance_epilogue(tol_pre, want, activation, out_kind)
        assert_within(got[sel], want, tol, f"group {z}")
    return got


def test_nvfp4_grouped_small_edge_cases():
    """Empty groups, -1 and out-of-range ids (zeros), a row before the first
    group and rows after the last (untouched), groups larger than one tile."""
    lib()
    q, bs, s2 = synth.nvfp4_expert_stack(3, 300, 128, seed=1)
    a = synth.bf16_activations(420, 128, seed=2)
    offs = [1, 130, 130, 200, 333, 333, 400]
    ids = [2, 0, -1, 1, 5, 0]
    run_grouped(a, q, bs, s2, offs, ids, max_rows=200)


def test_nvfp4_grouped_pair_tile_rows():
    """As the FP8 test: groups of 255 to 1100 rows over 512-row pair tiles."""
    lib()
    q, bs, s2 = synth.nvfp4_expert_stack(3, 300, 128, seed=11)
    sizes = [255, 256, 257, 511, 512, 513, 1100, 0, 1, 700]
    offs = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    ids = [0, 1, 2, 0, 1, -1, 2, 1, 0, 1]
    a = synth.bf16_activations(offs[-1], 128, seed=12)
    run_grouped(a, q, bs, s2, offs, ids, max_rows=max(sizes))


@pytest.mark.parametrize("k", [64, 192, 1024])
def test_nvfp4_grouped_k_multiples_of_64(k):
    """K a multiple of 64 but not of the 128-element k-step where it is odd."""
    lib()
    q, bs, s2 = synth.nvfp4_expert_stack(2, 264, k, seed=k)
    a = synth.bf16_activations(290, k, seed=k + 1)
    run_grouped(a, q, bs, s2, [0, 17, 290], [1, 0], max_rows=273, out_dtype=torch.bfloat16)


def test_nvfp4_grouped_raw_no_scales_f16():
    lib()
    q, bs, _ = synth.nvfp4_expert_stack(2, 256, 256, seed=3)
    a = synth.bf16_activations(300, 256, seed=4)
    run_grouped(a, q, bs, None, [0, 150, 300], [1, 0], max_rows=150, out_dtype=torch.float16)


@pytest.mark.parametrize("act", ["none", "relu", "silu", "gelu_tanh"])
def test_nvfp4_grouped_epilogue(act):
    """Bias [E, N] picked by the group's expert, then the activation; the
    zero groups stay zero (no bias)."""
    lib()
    q, bs, s2 = synth.nvfp4_expert_stack(3, 320, 256, seed=11)
    a = synth.bf16_activations(400, 256, seed=12)
    bias = (synth.gaussian((3, 320), 0.05, seed=13)).to(torch.bfloat16)
    run_grouped(a, q, bs, s2, [0, 90, 90, 250, 400], [2, 1, -1, 0], max_rows=160,
                out_dtype=torch.bfloat16, bias=bias, activation=act)


def test_nvfp4_grouped_moe_config_sampled():
    """8 experts [8, 14336, 4096], 4096 rows routed by the seeded multinomial
    (expert 3 empty, last group -1), checked on sampled rows of every group."""
    lib()
    q, bs, s2 = synth.nvfp4_expert_stack(8, 14336, 4096, seed=0)
    a = synth.bf16_activations(4096, 4096, seed=1)
    offs, ids, counts = synth.moe_routing(4096, seed=2)
    assert int(counts[3]) == 0 and int(ids[-1]) == -1
    rng = np.random.default_rng(5)
    rows = []
    for z in range(len(ids)):
        r0, r1 = int(offs[z]), int(offs[z + 1])
        if r1 > r0:
            rows += [r0, r1 - 1] + list(rng.integers(r0, r1, 4))
    rows = np.array(sorted(set(rows)))
    run_grouped(a, q, bs, s2, offs.numpy(), ids.numpy(), int(counts.max()),
                out_dtype=torch.bfloat16, rows=rows)


def test_nvfp4_grouped_equals_dense_per_group():
    """Each group's rows equal the dense NVFP4 product of its expert (the
    same kernel family, K = 512 in one split: bit-equal)."""
    lib()
    q, bs, s2 = synth.nvfp4_expert_stack(2, 384, 512, seed=6)
    a = synth.bf16_activations(520, 512, seed=7)
    offs, ids = [0, 200, 520], [1, 0]
    got = run_grouped(a, q, bs, s2, offs, ids, max_rows=320)
    for z, e in enumerate(ids):
        rows = a[offs[z]:offs[z + 1]]
        dense = to_f64(gq.nvfp4_matmul(rows.to(DEV), q[e].to(DEV), bs[e].to(DEV), float(s2[e]),
                                       out_dtype=torch.float32))
        tol = 2 * oracle.tolerance(bits(rows), oracle.decode_nvfp4(q[e].numpy(), bs[e].numpy()),
                                   float(s2[e]))
        assert_within(dense, got[offs[z]:offs[z + 1]], tol, f"group {z} vs dense")


def test_nvfp4_grouped_identity_exact():
    """a = I (K = 64 rows of the identity, one group per expert): every output
    element is one decoded weight times its expert's scale 1, exactly."""
    lib()
    k, n = 64, 256
    q, bs, _ = synth.nvfp4_expert_stack(2, n, k, seed=15)
    eye = torch.eye(k, dtype=torch.bfloat16)
    a = torch.cat([eye, eye])
    out = torch.full((2 * k, n), SENTINEL, dtype=torch.float32, device=DEV)
    gq.nvfp4_grouped_matmul(a.to(DEV), q.to(DEV), bs.to(DEV),
                            torch.tensor([0, k, 2 * k], dtype=torch.int32, device=DEV),
                            torch.tensor([1, 0], dtype=torch.int32, device=DEV), None,
                            max_rows_per_group=k, out=out)
    got = to_f64(out)
    assert_exact(got[:k], oracle.decode_nvfp4(q[1].numpy(), bs[1].numpy()).T, "expert 1",
                 signed_zero=False)
    assert_exact(got[k:], oracle.decode_nvfp4(q[0].numpy(), bs[0].numpy()).T, "expert 0",
                 signed_zero=False)


def test_nvfp4_grouped_rejects_bad_k():
    lib()
    l = gq.load_library()
    a = torch.zeros((4, 96), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    o = torch.zeros(4, dtype=torch.int32, device=DEV)
    c = torch.zeros((4, 32), dtype=torch.float32, device=DEV)
    st = l.gq_nvfp4_grouped_matmul(c.data_ptr(), 0, a.data_ptr(), w.data_ptr(), w.data_ptr(),
                                   o.data_ptr(), o.data_ptr(), None, 1, 1, 4, 4, 32, 96, None)
    assert st == 2  # GQ_ERR_SHAPE


def test_nvfp4_grouped_k_zero_writes_zeros():
    """K = 0: every covered row is an empty sum (zeros); uncovered rows stay."""
    lib()
    q = torch.zeros((2, 64, 0), dtype=torch.uint8, device=DEV)
    bs = torch.zeros((2, 64, 0), dtype=torch.uint8, device=DEV)
    a = torch.zeros((10, 0), dtype=torch.bfloat16, device=DEV)
    out = torch.full((10, 64), SENTINEL, dtype=torch.float32, device=DEV)
    gq.nvfp4_grouped_matmul(a, q, bs, torch.tensor([1, 5, 9], dtype=torch.int32, device=DEV),
                            torch.tensor([0, -1], dtype=torch.int32, device=DEV), None,
                            max_rows_per_group=8, out=out)
    got = out.cpu()
    assert torch.all(got[1:9] == 0.0)
    assert torch.all(got[0] == SENTINEL) and torch.all(got[9] == SENTINEL)
