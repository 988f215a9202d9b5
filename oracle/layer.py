"""The quantized linear layer, its grouped (MoE) form and materialize, float64.

Test infrastructure only (see the package docstring).

Definition followed (the "fp8_gemv" and "fp4_matmul" module pages, first
paragraphs): out = x @ dequant(W)^T with W stored [N, K] ("transpose_b"), so

    out[m, n] = alpha * sum_k x[m, k] * w_hat[n, k]

with x the bf16 activations taken exactly, w_hat the decoded weight
(``decode``) and alpha the per-tensor scale.  The "fp8_gemv" page, paragraph
"Scale contract", has the kernels produce the raw product and the per-tensor
``weight_scale`` (NVFP4: ``weight_scale_2``) folded as one multiply after the
sum, which is exact because a scalar factors out of the sum; here alpha is
applied to the float64 sum, alpha = 1 is the raw product.  The bf16
``input_scale`` cancels for bf16 activations (same paragraph), so there is none.

The grouped form follows the "Matmul2dFp8" page, method ``run_grouped``: for
group z the rows a_offsets[z] .. a_offsets[z+1]-1 of A are multiplied with the
weight of expert expert_ids[z]; a group with no rows does nothing; a group whose
expert id is -1 writes zeros to its rows; the per-expert scale is folded after
the product like the per-tensor one.

The float64 sums use numpy's matmul (a library primitive standing in for the
sum); ``linear_loops`` is the same definition as three plain loops, for tiny
shapes and for checking the numpy route.
"""

import math

import numpy as np

from .decode import decode_fp8, decode_nvfp4
from .formats import bf16_bits_to_f64, f16_bits_to_f64


def _activations(x) -> np.ndarray:
    """Activations as float64: uint16 input is taken as bfloat16 bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


def linear(x, w_hat, alpha=1.0) -> np.ndarray:
    """alpha * x @ w_hat^T in float64.  x [M, K] (or [K]), w_hat [N, K]."""
    xf = _activations(x)
    w = np.asarray(w_hat, dtype=np.float64)
    return float(alpha) * (xf @ w.T)


def linear_loops(x, w_hat, alpha=1.0) -> np.ndarray:
    """The same product as three explicit loops (tiny shapes only)."""
    xf = np.atleast_2d(_activations(x))
    w = np.asarray(w_hat, dtype=np.float64)
    m_rows, k_len = xf.shape
    n_rows = w.shape[0]
    out = np.zeros((m_rows, n_rows), dtype=np.float64)
    for m in range(m_rows):
        for n in range(n_rows):
            acc = 0.0
            for k in range(k_len):
                acc += float(xf[m, k]) * float(w[n, k])
            out[m, n] = float(alpha) * acc
    return out


def fp8_gemv(x, w_codes, alpha=1.0) -> np.ndarray:
    """M = 1 FP8 GEMV: x [K] (bf16), W [N, K] e4m3 codes -> float64 [N]."""
    xf = _activations(x).reshape(-1)
    return linear(xf[None, :], decode_fp8(w_codes), alpha)[0]


def fp8_matmul(a, w_codes, alpha=1.0) -> np.ndarray:
    """FP8 GEMM: A [M, K] (bf16), W [N, K] e4m3 codes -> float64 [M, N]."""
    return linear(a, decode_fp8(w_codes), alpha)


def nvfp4_gemv(x, q_packed, block_scales, alpha=1.0) -> np.ndarray:
    """M = 1 NVFP4 GEMV -> float64 [N]; alpha is the per-tensor second scale."""
    xf = _activations(x).reshape(-1)
    return linear(xf[None, :], decode_nvfp4(q_packed, block_scales), alpha)[0]


def nvfp4_matmul(a, q_packed, block_scales, alpha=1.0) -> np.ndarray:
    """NVFP4 GEMM: A [M, K] (bf16) -> float64 [M, N]."""
    return linear(a, decode_nvfp4(q_packed, block_scales), alpha)


def _grouped(a, n_experts, n_cols, decode_expert, a_offsets, expert_ids, expert_scales, rows):
    """The grouped loop of ``run_grouped``, with the weight of expert e given by
    decode_expert(e) (float64 [N, K])."""
    offs = [int(v) for v in np.asarray(a_offsets).reshape(-1)]
    ids = [int(v) for v in np.asarray(expert_ids).reshape(-1)]
    a_arr = np.asarray(a)
    total_m = a_arr.shape[0]
    out = np.full((total_m, n_cols), np.nan, dtype=np.float64)
    written = np.zeros(total_m, dtype=bool)
    wanted = None if rows is None else np.zeros(total_m, dtype=bool)
    if wanted is not None:
        wanted[np.asarray(rows, dtype=np.int64)] = True
    decoded = {}
    for z, expert in enumerate(ids):
        start, stop = offs[z], offs[z + 1]
        if stop <= start:
            continue                      # empty group: nothing to do
        sel = np.arange(start, stop)
        if wanted is not None:
            sel = sel[wanted[sel]]
        if sel.size == 0:
            written[start:stop] = True
            continue
        if expert == -1 or not (0 <= expert < n_experts):
            out[sel, :] = 0.0             # inactive group writes zeros
        else:
            if expert not in decoded:
                decoded[expert] = decode_expert(expert)
            scale = 1.0 if expert_scales is None else float(np.asarray(expert_scales)[expert])
            out[sel, :] = linear(a_arr[sel], decoded[expert], scale)
        written[start:stop] = True
    return out, written


def fp8_grouped_matmul(a, w_stack, a_offsets, expert_ids, expert_scales=None,
                       rows=None):
    """Grouped (MoE) FP8 product.

    a:             [total_M, K] activations (bf16 bits or float values)
    w_stack:       uint8 [E, N, K] e4m3 codes, one weight per expert
    a_offsets:     [G + 1] row offsets; group z owns rows a_offsets[z] .. a_offsets[z+1]-1
    expert_ids:    [G] expert of each group; -1 marks a group that writes zeros
    expert_scales: [E] per-expert scale folded after the product, or None (raw)
    rows:          optional sorted array of row indices to compute (others are
                   left NaN); used to check a few rows of a large problem.

    Returns (out [total_M, N] float64, written [total_M] bool).  Rows that no
    group covers are NaN and not marked written.
    """
    w_stack = np.asarray(w_stack, dtype=np.uint8)
    n_experts, n_cols, _ = w_stack.shape
    return _grouped(a, n_experts, n_cols, lambda e: decode_fp8(w_stack[e]), a_offsets,
                    expert_ids, expert_scales, rows)


def nvfp4_grouped_matmul(a, q_stack, bs_stack, a_offsets, expert_ids, expert_scales=None,
                         rows=None):
    """Grouped (MoE) NVFP4 product: the same groups as ``fp8_grouped_matmul``
    with expert e's weight the NVFP4 pair q_stack[e] (uint8 [N, K/2]) and
    bs_stack[e] (uint8 [N, K/16]); expert_scales[e] is its second scale."""
    q_stack = np.asarray(q_stack, dtype=np.uint8)
    bs_stack = np.asarray(bs_stack, dtype=np.uint8)
    n_experts, n_cols, _ = q_stack.shape
    return _grouped(a, n_experts, n_cols, lambda e: decode_nvfp4(q_stack[e], bs_stack[e]),
                    a_offsets, expert_ids, expert_scales, rows)


def fp8_materialize(w_codes) -> np.ndarray:
    """Dense decoded FP8 weight [N, K], float64, no scale applied."""
    return decode_fp8(w_codes)


def nvfp4_materialize(q_packed, block_scales) -> np.ndarray:
    """Dense decoded NVFP4 weight [N, K], float64, no per-tensor scale applied."""
    return decode_nvfp4(q_packed, block_scales)


def abs_dot(x, w_hat, alpha=1.0) -> np.ndarray:
    """|alpha| * sum_k |x_k * w_hat_k| for every output: the size of the sum,
    the quantity the floating-point tolerance is relative to."""
    xf = np.abs(_activations(x))
    w = np.abs(np.asarray(w_hat, dtype=np.float64))
    if xf.ndim == 1:
        xf = xf[None, :]
    return abs(float(alpha)) * (xf @ w.T)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bfloat16 numbers at |v| (2^(e-7) for |v| in [2^e, 2^(e+1)),
    2^-133 below the smallest normal)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(np.isfinite(a), a, 0.0))
    ulp = np.ldexp(1.0, (e - 1 - 7).astype(np.int64))
    return np.where((a < 2.0 ** -126) | ~np.isfinite(a), 2.0 ** -133, ulp)


def tolerance(x, w_hat, alpha=1.0, out_bf16=False, ref=None) -> np.ndarray:
    """Allowed |gpu - oracle| per output: 2e-4 * |alpha| * sum_k |x_k w_k|,
    plus one bfloat16 ulp of the result when the output is stored as bf16."""
    tol = 2e-4 * abs_dot(x, w_hat, alpha)
    if out_bf16:
        if ref is None:
            ref = linear(x, w_hat, alpha)
        tol = tol + bf16_ulp(np.abs(ref) + tol)
    return tol


# ------------------------------------------------------------------ epilogue --
#
# The "Matmul2dFp8" struct page gives the tiled matmul an optional fused
# epilogue: an elementwise function of the output coordinate (row, col) and
# the computed value, applied where the result is stored.  The layer's
# epilogue, in the order a linear layer applies it, is
#
#     out[m, n] = act(alpha * sum_k x[m, k] w_hat[n, k] + bias[n])
#
# (grouped: the bias row of the group's expert), with act one of the
# activations below, written from their definitions.

def f16_ulp(v) -> np.ndarray:
    """Spacing of binary16 numbers at |v| (2^(e-10) for |v| in [2^e, 2^(e+1)),
    2^-24 below the smallest normal 2^-14)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(np.isfinite(a), a, 0.0))
    ulp = np.ldexp(1.0, (e - 1 - 10).astype(np.int64))
    return np.where((a < 2.0 ** -14) | ~np.isfinite(a), 2.0 ** -24, ulp)


def activation(v, kind: str) -> np.ndarray:
    """Elementwise activation, float64.

    none:      v
    relu:      v for v > 0, else 0 (NaN stays NaN)
    silu:      v / (1 + exp(-v))                      (v times the logistic sigmoid)
    gelu_tanh: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))   (tanh form of GELU)
    """
    v = np.asarray(v, dtype=np.float64)
    if kind == "none":
        return v.copy()
    if kind == "relu":
        return np.where(v > 0, v, np.where(np.isnan(v), v, 0.0))
    if kind == "silu":
        with np.errstate(over="ignore", invalid="ignore"):
            return v / (1.0 + np.exp(-v))
    if kind == "gelu_tanh":
        c = math.sqrt(2.0 / math.pi)
        with np.errstate(over="ignore", invalid="ignore"):
            return 0.5 * v * (1.0 + np.tanh(c * (v + 0.044715 * v ** 3)))
    raise ValueError(f"unknown activation {kind!r}")


# Upper bounds of |d act / dv| over the reals: how far an error in the
# pre-activation value can move the output.
ACT_LIPSCHITZ = {"none": 1.0, "relu": 1.0, "silu": 1.1, "gelu_tanh": 1.13}


def epilogue(v, bias=None, act: str = "none") -> np.ndarray:
    """act(v + bias) with bias broadcast along the last axis (the column n)."""
    v = np.asarray(v, dtype=np.float64)
    if bias is not None:
        v = v + np.asarray(bias, dtype=np.float64)
    return activation(v, act)


def tolerance_epilogue(tol_pre, ref_out, act: str = "none", out_kind: str = "f32") -> np.ndarray:
    """Allowed |gpu - oracle| after the epilogue.

    tol_pre is the allowed error of the pre-activation value (``tolerance``
    without the output rounding).  The activation moves it by at most its
    Lipschitz bound; the fp32 bias add and the fp32 activation functions add
    a few units in the last place of the fp32 result (2^-20 |out| covers
    them); the output conversion adds one unit in the last place of the
    output type.
    """
    ref = np.abs(np.asarray(ref_out, dtype=np.float64))
    tol = ACT_LIPSCHITZ[act] * np.asarray(tol_pre, dtype=np.float64) + 2.0 ** -20 * ref
    if out_kind == "bf16":
        tol = tol + bf16_ulp(ref + tol)
    elif out_kind == "f16":
        tol = tol + f16_ulp(ref + tol)
    return tol
