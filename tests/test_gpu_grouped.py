"""Grouped (MoE) FP8 GEMM against the oracle's per-group definition."""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_within, bits, lib, to_f64

pytestmark = pytest.mark.gpu

SENTINEL = -7.25


def run_grouped(a, stack, scales, offs, ids, max_rows, out_dtype=torch.float32, rows=None):
    total_m = a.shape[0]
    n = stack.shape[1]
    out = torch.full((total_m, n), SENTINEL, dtype=out_dtype, device=DEV)
    gq.fp8_grouped_matmul(a.to(DEV), stack.to(DEV), torch.as_tensor(offs, dtype=torch.int32).to(DEV),
                          torch.as_tensor(ids, dtype=torch.int32).to(DEV),
                          None if scales is None else scales.to(DEV),
                          max_rows_per_group=max_rows, out=out)
    torch.cuda.synchronize()
    got = to_f64(out)
    ab = bits(a)
    ref, written = oracle.fp8_grouped_matmul(ab, stack.numpy(), np.asarray(offs), np.asarray(ids),
                                             None if scales is None else scales.numpy(), rows=rows)
    # rows no group covers stay untouched
    assert np.all(got[~written] == SENTINEL)
    # per group tolerance
    offs = np.asarray(offs)
    for z, e in enumerate(np.asarray(ids)):
        r0, r1 = int(offs[z]), int(offs[z + 1])
        if r1 <= r0:
            continue
        sel = np.arange(r0, r1) if rows is None else np.intersect1d(np.arange(r0, r1), rows)
        if sel.size == 0:
            continue
        if e < 0 or e >= stack.shape[0]:
            assert np.all(got[sel] == 0.0), f"group {z} (id {e}) must be zero"
            continue
        w_hat = oracle.decode_fp8(stack[e].numpy())
        s = 1.0 if scales is None else float(scales[e])
        tol = oracle.tolerance(ab[sel], w_hat, s, out_dtype == torch.bfloat16, ref=ref[sel])
        assert_within(got[sel], ref[sel], tol, f"group {z}")
    return got


def test_grouped_small_edge_cases():
    """Empty groups, -1 and out-of-range ids (zeros), a row before the first
    group and rows after the last (untouched), groups larger than one tile."""
    lib()
    stack, scales = synth.fp8_expert_stack(3, 300, 128, seed=1)
    a = synth.bf16_activations(420, 128, seed=2)
    offs = [1, 130, 130, 200, 333, 333, 400]
    ids = [2, 0, -1, 1, 5, 0]
    run_grouped(a, stack, scales, offs, ids, max_rows=200)


def test_grouped_pair_tile_rows():
    """Groups of 255 to 1100 rows: one or both 256-row halves of a 512-row
    pair tile, and groups over several pair tiles with ragged tails; N with
    the odd CTA's weight rows partly past the end."""
    lib()
    stack, scales = synth.fp8_expert_stack(3, 300, 128, seed=11)
    sizes = [255, 256, 257, 511, 512, 513, 1100, 0, 1, 700]
    offs = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    ids = [0, 1, 2, 0, 1, -1, 2, 1, 0, 1]
    a = synth.bf16_activations(offs[-1], 128, seed=12)
    run_grouped(a, stack, scales, offs, ids, max_rows=max(sizes))


def test_grouped_raw_no_scales_bf16():
    lib()
    stack, _ = synth.fp8_expert_stack(2, 256, 256, seed=3)
    a = synth.bf16_activations(300, 256, seed=4)
    run_grouped(a, stack, None, [0, 150, 300], [1, 0], max_rows=150, out_dtype=torch.bfloat16)


def test_grouped_moe_config_sampled():
    """8 experts [8, 14336, 4096], 4096 rows routed by the seeded multinomial
    (expert 3 empty, last group -1), checked on sampled rows of every group."""
    lib()
    stack, scales = synth.fp8_expert_stack(8, 14336, 4096, seed=0)
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
    run_grouped(a, stack, scales, offs.numpy(), ids.numpy(), int(counts.max()),
                out_dtype=torch.bfloat16, rows=rows)


def test_grouped_equals_dense_per_group():
    lib()
    stack, scales = synth.fp8_expert_stack(2, 384, 512, seed=6)
    a = synth.bf16_activations(260, 512, seed=7)
    offs, ids = [0, 100, 260], [1, 0]
    got = run_grouped(a, stack, scales, offs, ids, max_rows=160)
    for z, e in enumerate(ids):
        rows = a[offs[z]:offs[z + 1]]
        dense = to_f64(gq.fp8_matmul(rows.to(DEV), stack[e].to(DEV),
                                     float(scales[e]), out_dtype=torch.float32))
        # Both sum exact products in fp32 in their own fixed order (the dense
        # call may split K): equal within twice the stated tolerance.
        tol = 2 * oracle.tolerance(bits(rows), oracle.decode_fp8(stack[e].numpy()), float(scales[e]))
        assert_within(dense, got[offs[z]:offs[z + 1]], tol, f"group {z} vs dense")


def test_grouped_max_rows_clips():
    """Rows past max_rows_per_group in a group are not computed (out of
    contract) and nothing outside the groups is written."""
    lib()
    stack, scales = synth.fp8_expert_stack(1, 256, 64, seed=8)
    a = synth.bf16_activations(300, 64, seed=9)
    out = torch.full((300, 256), SENTINEL, dtype=torch.float32, device=DEV)
    gq.fp8_grouped_matmul(a.to(DEV), stack.to(DEV), torch.tensor([0, 300], dtype=torch.int32, device=DEV),
                          torch.tensor([0], dtype=torch.int32, device=DEV), scales.to(DEV),
                          max_rows_per_group=130, out=out)
    got = to_f64(out)
    assert np.all(got[130:] == SENTINEL)
    assert not np.any(got[:130] == SENTINEL)
