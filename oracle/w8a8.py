"""W8A8 int8 linear layer: per-row activation quantization, and the
int8 x int8 product with its dequant epilogue.

Test infrastructure only (see the package docstring).

Source: the "int8_matmul" module page (Apple M5 int8 W8A8 matmul), which
computes out = dequant(A_int8 @ B_int8^T):

* both operands are symmetric-absmax int8 with scale = absmax / 127, A per
  row (per token), B per column (per output channel, i.e. per row of the
  [N, K] weight);
* A is quantized online by a separate one-pass kernel
  (enqueue_apple_int8_quantize_activation: int8 codes + an fp32 scale per
  row); B is quantized once, when the weight is loaded;
* the int8 products are summed exactly (int32 accumulation), then every
  output element is multiplied by a_scale[row] * b_scale[col], an optional
  per-column bias is added after the dequant, and the result is cast to the
  output type (bf16).

Readings where the page is silent (the kernel's precision decides):

* quantizer, in float32: absmax of the row's values, scale = absmax / 127
  (IEEE float32 division), code = round(x / scale) with float32 division and
  round-half-to-even, clamped to [-127, 127]; a row of zeros has scale 0 and
  codes 0 (the division is not evaluated);
* dequant, in float32 and in this order: (float32(acc) * a_scale[m]) *
  b_scale[n], then + bias[n], then one rounding to the output type; acc is
  the exact integer sum, converted to float32 with round-to-nearest-even.
  An activation (the shared fused epilogue) is applied after the bias.
"""

import numpy as np

from .formats import bf16_bits_to_f64

F32 = np.float32


def _as_values(x) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values; float arrays pass."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


def int8_quantize_rows(x):
    """Per-row symmetric absmax quantization of activations.

    x: [M, K] bf16 bit patterns (or float values exactly representable in
       float32).
    Returns (q int8 [M, K], scale float32 [M]).
    """
    xf = _as_values(x).astype(F32)                 # exact: bf16 is a subset of float32
    if xf.ndim != 2:
        raise ValueError("x must be [M, K]")
    m, k = xf.shape
    absmax = np.max(np.abs(xf), axis=1) if k else np.zeros(m, dtype=F32)
    scale = (absmax.astype(F32) / F32(127.0)).astype(F32)
    q = np.zeros((m, k), dtype=np.int8)
    nz = scale > 0
    if np.any(nz):
        ratio = (xf[nz] / scale[nz][:, None]).astype(F32)   # float32 division
        q[nz] = np.clip(np.rint(ratio), -127, 127).astype(np.int8)   # ties to even
    return q, scale


def int8_accumulate(q_a, q_b) -> np.ndarray:
    """Exact integer sums acc[m, n] = sum_k q_a[m, k] * q_b[n, k] (int64)."""
    a = np.asarray(q_a, dtype=np.int8).astype(np.int64)
    b = np.asarray(q_b, dtype=np.int8).astype(np.int64)
    return a @ b.T


def int8_dequant(acc, a_scale, b_scale, bias=None) -> np.ndarray:
    """float32 dequant of the exact sums: (f32(acc) * a_scale[m]) * b_scale[n]
    (+ bias[n]), each step rounded to float32.  Returns float32 [M, N]."""
    accf = np.asarray(acc).astype(F32)             # round-to-nearest-even from int64
    sa = np.asarray(a_scale, dtype=F32)[:, None]
    sb = np.asarray(b_scale, dtype=F32)[None, :]
    v = (accf * sa).astype(F32)
    v = (v * sb).astype(F32)
    if bias is not None:
        v = (v + _as_values(bias).astype(F32)[None, :]).astype(F32)
    return v


def int8_matmul(q_a, q_b, a_scale, b_scale, bias=None) -> np.ndarray:
    """The W8A8 product before the output cast: float32 [M, N]."""
    return int8_dequant(int8_accumulate(q_a, q_b), a_scale, b_scale, bias)


def int8_abs_sum(q_a, q_b) -> np.ndarray:
    """sum_k |q_a[m, k] * q_b[n, k]| per output: a float32 accumulator adding
    the products in any order holds every partial sum exactly (and so gives
    the exact integer result) where this is below 2^24."""
    a = np.abs(np.asarray(q_a, dtype=np.int8).astype(np.int64))
    b = np.abs(np.asarray(q_b, dtype=np.int8).astype(np.int64))
    return a @ b.T
