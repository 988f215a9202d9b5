"""Failure detection without a GPU fault: a bounded in-kernel wait that runs
out is reported in the device status word, the kernel unwinds, and the
context stays usable.

GQ_LAUNCH_TEST_STALL_PRODUCER makes the tensor-core GEMM's copy producer
issue nothing, so no shared-memory stage ever fills and the waits of the
MMA, dequant and epilogue roles run out after the short limit set with
gq_set_wait_limit_ns.  Nothing asynchronous (copy, MMA, store) is in flight
when the CTAs exit.  Each test checks that the call returns promptly, that
the status word names only timed-out consumer roles, that the reset clears
it, that the output was left as it was, and that the next normal call on the
same context is correct.
"""

import time

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_within, bits, lib, to_f64

pytestmark = pytest.mark.gpu

# status bits (common.cuh): producer, MMA, dequant, epilogue, other
PRODUCER, MMA, DEQUANT, EPILOGUE = 1, 2, 4, 8
LIMIT_NS = 1_000_000      # 1 ms


def stalled(call):
    """Run `call` with the producer stalled and a 1 ms wait limit; returns the
    seconds until the device was idle again and the status word it left."""
    torch.cuda.synchronize()
    assert gq.device_status(reset=True) == 0
    gq.set_wait_limit_ns(LIMIT_NS)
    gq.set_launch_flags(gq.GQ_LAUNCH_TEST_STALL_PRODUCER)
    try:
        t0 = time.time()
        call()
        torch.cuda.synchronize()
        dt = time.time() - t0
    finally:
        gq.set_launch_flags(0)
        gq.set_wait_limit_ns(0)
    return dt, gq.device_status()


def check_recovered(st):
    assert st != 0, "no wait reported a time-out"
    assert st & ~(MMA | DEQUANT | EPILOGUE) == 0, f"unexpected status bits {st:#x}"
    assert gq.device_status(reset=True) == st
    assert gq.device_status() == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_stalled_producer_times_out_and_recovers(fmt):
    lib()
    m, n, k = 300, 256, 128          # M > 128: the persistent tensor-core GEMM, 2 tiles
    a = synth.bf16_activations(m, k, seed=4)
    out = torch.full((m, n), 7.25, dtype=torch.float32, device=DEV)
    if fmt == "fp8":
        codes, s = synth.fp8_weight(n, k, seed=3)
        w_hat = oracle.decode_fp8(codes.numpy())
        run = lambda o: gq.fp8_matmul(a.to(DEV), codes.to(DEV), s, out=o)
    else:
        q, bs, s = synth.nvfp4_weight(n, k, seed=3)
        w_hat = oracle.decode_nvfp4(q.numpy(), bs.numpy())
        run = lambda o: gq.nvfp4_matmul(a.to(DEV), q.to(DEV), bs.to(DEV), s, out=o)
    dt, st = stalled(lambda: run(out))
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    check_recovered(st)
    assert torch.all(out == 7.25), "a stalled GEMM wrote its output"
    # the same context computes the next call correctly
    c = torch.empty((m, n), dtype=torch.float32, device=DEV)
    run(c)
    torch.cuda.synchronize()
    ab = bits(a)
    ref = oracle.linear(ab, w_hat, s)
    assert_within(to_f64(c), ref, oracle.tolerance(ab, w_hat, s), f"{fmt} gemm after time-out")
    assert gq.device_status() == 0


def test_stalled_w8a8_split_k_times_out_and_recovers():
    """The W8A8 GEMM with K split over a cluster (M = 5, K = 16384): every CTA
    of the cluster times out, none adds a partial, all leave the cluster
    barriers, and the next call is bit-exact."""
    lib()
    m, n, k = 5, 256, 16384
    qa, sa = synth.int8_codes(m, k, seed=21)
    qb, sb = synth.int8_weight(n, k, seed=22)
    out = torch.full((m, n), 7.25, dtype=torch.float32, device=DEV)
    run = lambda o: gq.int8_matmul(qa.to(DEV), qb.to(DEV), sa.to(DEV), sb.to(DEV), out=o)
    dt, st = stalled(lambda: run(out))
    assert dt < 5.0
    check_recovered(st)
    assert torch.all(out == 7.25)
    c = torch.empty((m, n), dtype=torch.float32, device=DEV)
    run(c)
    torch.cuda.synchronize()
    want = oracle.int8_matmul(qa.numpy(), qb.numpy(), sa.numpy(), sb.numpy())
    assert np.array_equal(c.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert gq.device_status() == 0


@pytest.mark.parametrize("k", [100, 33, 104])
def test_stalled_anyk_times_out_and_recovers(k):
    """The FP8 GEMM with K % 16 != 0 on CTA pairs (M > 256): K = 100 realigns A
    in two residue classes whose rows span several dequant warps (their
    named barrier also votes on a failed wait), K = 33 in eight classes of
    one warp each, K = 104 takes A by the tiled box.  Every role's wait runs
    out, all leave together, and the next call is correct."""
    lib()
    m, n = 300, 256
    a = synth.bf16_activations(m, k, seed=5)
    codes, s = synth.fp8_weight(n, k, seed=6)
    w_hat = oracle.decode_fp8(codes.numpy())
    out = torch.full((m, n), 7.25, dtype=torch.float32, device=DEV)
    run = lambda o: gq.fp8_matmul(a.to(DEV), codes.to(DEV), s, out=o)
    dt, st = stalled(lambda: run(out))
    assert dt < 5.0, f"the stalled call took {dt:.2f} s"
    check_recovered(st)
    assert torch.all(out == 7.25), "a stalled GEMM wrote its output"
    c = torch.empty((m, n), dtype=torch.float32, device=DEV)
    run(c)
    torch.cuda.synchronize()
    ab = bits(a)
    ref = oracle.linear(ab, w_hat, s)
    assert_within(to_f64(c), ref, oracle.tolerance(ab, w_hat, s), f"any-K {k} after time-out")
    assert gq.device_status() == 0
