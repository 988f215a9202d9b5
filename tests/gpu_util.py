"""Helpers for the GPU parity tests: load the library (failing loudly if it
is missing), move seeded inputs to the GPU, and compare GPU outputs with the
CPU oracle element by element."""

from __future__ import annotations

import numpy as np
import torch

import gemm_fp8_nvfp4_gb300 as gq
import oracle
import synth

DEV = "cuda:0"


def lib():
    """The CUDA library must be there on a GPU run: no skip, no fallback."""
    return gq.load_library()


def to_f64(t: torch.Tensor) -> np.ndarray:
    """GPU output (float32, bf16 or f16) -> float64 numpy, exactly (the 16-bit
    types decoded from their bit patterns by the oracle's format code)."""
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    if t.dtype == torch.float16:
        return oracle.f16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    return t.to(torch.float64).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def assert_exact(got: np.ndarray, want: np.ndarray, what="", signed_zero=True):
    """Bit-exact comparison of values: equal values, equal sign of zero, NaN
    exactly where the oracle has NaN (any NaN payload).  signed_zero=False
    accepts +0 for -0: used where the result is an IEEE sum whose exact value
    is zero (x + (-0) with x = +0 is +0)."""
    assert got.shape == want.shape, (got.shape, want.shape)
    gn, wn = np.isnan(got), np.isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ at {np.argwhere(gn != wn)[:5]}"
    m = ~wn
    bad = got[m] != want[m]
    if signed_zero:
        bad |= np.signbit(got[m]) != np.signbit(want[m])
    if bad.any():
        idx = np.argwhere(m)[np.nonzero(bad)[0][:5]]
        raise AssertionError(f"{what}: {bad.sum()} values differ, first at {idx.tolist()}: "
                             f"got {got[tuple(idx[0])]}, want {want[tuple(idx[0])]}")


def assert_within(got: np.ndarray, ref: np.ndarray, tol: np.ndarray, what=""):
    """|got - ref| <= tol element by element; NaN must match NaN."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    m = ~rn
    err = np.abs(got[m] - ref[m])
    t = np.broadcast_to(tol, ref.shape)[m]
    bad = err > t
    if bad.any():
        i = int(np.argmax(err - t))
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst "
                             f"err {err[i]:.3e} vs tol {t[i]:.3e} (ref {ref[m][i]:.6e})")


def canary_out(shape, dtype, pad=64, fill=-7.25):
    """An output tensor embedded in a larger buffer filled with a sentinel, to
    check that the kernel writes nothing outside it."""
    n = int(np.prod(shape))
    buf = torch.full((pad + n + pad,), fill, dtype=dtype, device=DEV)
    return buf, buf[pad:pad + n].view(*shape)


def assert_canary(buf, pad=64, fill=-7.25):
    head = buf[:pad].float().cpu()
    tail = buf[-pad:].float().cpu()
    assert torch.all(head == fill) and torch.all(tail == fill), "write outside the output"
