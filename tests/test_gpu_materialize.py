"""Materialize kernels against the oracle: bit-exact on every code."""

import numpy as np
import pytest
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth
from tests.gpu_util import DEV, assert_canary, assert_exact, canary_out, lib, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n,k", [(1, 256), (7, 269), (33, 1024), (3, 5), (1, 1)])
def test_fp8_materialize_all_codes(n, k, out_dtype):
    lib()
    codes = (np.arange(n * k) * 37 % 256).astype(np.uint8).reshape(n, k)
    w = torch.from_numpy(codes).to(DEV)
    buf, out = canary_out((n, k), out_dtype)
    gq.fp8_materialize(w, out=out)
    torch.cuda.synchronize()
    assert_exact(to_f64(out), oracle.fp8_materialize(codes), "fp8 materialize")
    assert_canary(buf)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_nvfp4_materialize_all_code_scale_pairs(out_dtype):
    lib()
    # every (E2M1 code, E4M3 scale) pair: 256 rows (one scale code each),
    # 16 elements per block, each block holding all 16 E2M1 codes.
    n, k = 256, 64
    nib = np.tile(np.arange(16, dtype=np.uint8), k // 16)
    rows = []
    for r in range(n):
        rot = np.roll(nib, r % 16)
        rows.append(rot[0::2] | (rot[1::2] << 4))
    q = np.stack(rows).astype(np.uint8)
    bs = np.repeat(np.arange(256, dtype=np.uint8)[:, None], k // 16, axis=1)
    bs[:, 1] = ((bs[:, 1].astype(np.int32) + 91) % 256).astype(np.uint8)
    buf, out = canary_out((n, k), out_dtype)
    gq.nvfp4_materialize(torch.from_numpy(q).to(DEV), torch.from_numpy(bs).to(DEV), out=out)
    torch.cuda.synchronize()
    assert_exact(to_f64(out), oracle.nvfp4_materialize(q, bs), "nvfp4 materialize")
    assert_canary(buf)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_materialize_seeded_weights(out_dtype):
    lib()
    codes, _ = synth.fp8_weight(300, 512, seed=0)
    got = gq.fp8_materialize(codes.to(DEV), out_dtype=out_dtype)
    assert_exact(to_f64(got), oracle.fp8_materialize(codes.numpy()), "fp8")
    q, bs, _ = synth.nvfp4_weight(300, 512, seed=0)
    got = gq.nvfp4_materialize(q.to(DEV), bs.to(DEV), out_dtype=out_dtype)
    assert_exact(to_f64(got), oracle.nvfp4_materialize(q.numpy(), bs.numpy()), "nvfp4")


def test_materialize_errors():
    l = lib()
    w = torch.zeros(4, 16, dtype=torch.uint8, device=DEV)
    out = torch.empty(4, 16, dtype=torch.float32, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    assert l.gq_fp8_materialize(out.data_ptr(), 0, None, 4, 16, s) == 1          # NULL
    assert l.gq_fp8_materialize(out.data_ptr(), 0, w.data_ptr(), -1, 16, s) == 2  # shape
    assert l.gq_fp8_materialize(out.data_ptr(), 9, w.data_ptr(), 4, 16, s) == 4   # dtype
    assert l.gq_fp8_materialize(out.data_ptr() + 4, 0, w.data_ptr(), 4, 8, s) == 3  # align
    assert l.gq_nvfp4_materialize(out.data_ptr(), 0, w.data_ptr(), w.data_ptr(), 4, 24, s) == 2
    assert l.gq_fp8_materialize(out.data_ptr(), 0, w.data_ptr(), 0, 16, s) == 0   # empty
