"""Plant plausible mistakes in the oracle (on the CPU) and show that the pins
catch each one: a pin that no mistake can fail would pin nothing.

Each mutation patches one oracle function for the duration of one test; the
assertion is that at least one check in ``pins.ALL_CHECKS`` fails.
"""

import math

import numpy as np
import pytest

import oracle
import oracle.decode
import oracle.formats
import oracle.layer
import oracle.w8a8
from tests import pins


def _any_check_fails():
    for check in pins.ALL_CHECKS:
        try:
            check(oracle)
        except AssertionError:
            return check.__name__
        except Exception:  # a crash under the mutation also counts as caught
            return check.__name__
    return None


def _e4m3_wrong_bias(code):
    s, e, m = (code >> 7) & 1, (code >> 3) & 0xF, code & 7
    if e == 0xF and m == 7:
        return math.nan
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 8)
    return -mag if s else mag


def _e4m3_no_subnormal(code):
    s, e, m = (code >> 7) & 1, (code >> 3) & 0xF, code & 7
    if e == 0xF and m == 7:
        return math.nan
    mag = 0.0 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def _e2m1_sign_bit2(code):
    s, e, m = (code >> 2) & 1, (code >> 1) & 1, code & 1
    mag = m * 0.5 if e == 0 else (1 + m / 2.0)
    return -mag if s else mag


def _nvfp4_high_nibble_first(q, bs):
    q = np.asarray(q, dtype=np.uint8)
    swapped = ((q & 0xF) << 4) | (q >> 4)
    return ORIG_DECODE_NVFP4(swapped.astype(np.uint8), bs)


def _nvfp4_block_of_8(q, bs):
    q = np.asarray(q, dtype=np.uint8)
    bs = np.asarray(bs, dtype=np.uint8)
    n, half = q.shape
    k = 2 * half
    codes = np.empty((n, k), dtype=np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    t4, t8 = oracle.e2m1_table(), oracle.e4m3_table()
    idx = np.minimum(np.arange(k) // 8, bs.shape[1] - 1)
    return t4[codes] * t8[bs][:, idx]


def _linear_no_transpose(x, w_hat, alpha=1.0):
    xf = oracle.layer._activations(x)
    w = np.asarray(w_hat, dtype=np.float64)
    if xf.shape[-1] == w.shape[0] and w.shape[0] == w.shape[1]:
        return float(alpha) * (xf @ w)
    return float(alpha) * (xf @ w[:, ::-1].T)


def _linear_drop_alpha(x, w_hat, alpha=1.0):
    return ORIG_LINEAR(x, w_hat, 1.0)


def _linear_abs_weights(x, w_hat, alpha=1.0):
    return ORIG_LINEAR(x, np.abs(w_hat), alpha)


def _linear_drop_last_k(x, w_hat, alpha=1.0):
    xf = oracle.layer._activations(x)
    w = np.asarray(w_hat, dtype=np.float64)
    return float(alpha) * (xf[..., :-1] @ w[:, :-1].T)


def _f16_ties_away(x: float) -> int:
    # round half away from zero instead of to even
    import math
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if math.isnan(a) or math.isinf(a) or a == 0.0:
        return ORIG_F16(x)
    m, e = math.frexp(a)
    q_exp = max(e - 1, -14) - 10
    n = math.floor(math.ldexp(a, -q_exp) + 0.5)
    return ORIG_F16(math.copysign(math.ldexp(n, q_exp), -1.0 if sign else 1.0))


def _gelu_wrong_constant(v, kind):
    if kind == "gelu_tanh":
        v = np.asarray(v, dtype=np.float64)
        c = (2.0 / np.pi) ** 0.5
        return 0.5 * v * (1.0 + np.tanh(c * (v + 0.0447 * v ** 2)))
    return ORIG_ACT(v, kind)


def _silu_wrong_sign(v, kind):
    if kind == "silu":
        v = np.asarray(v, dtype=np.float64)
        with np.errstate(over="ignore"):
            return v / (1.0 + np.exp(v))
    return ORIG_ACT(v, kind)


def _epilogue_act_first(v, bias=None, act="none"):
    out = oracle.layer.activation(v, act)
    return out if bias is None else out + np.asarray(bias, dtype=np.float64)


def _int8_quant_ties_away(x):
    xf = oracle.w8a8._as_values(x).astype(np.float32)
    absmax = np.max(np.abs(xf), axis=1)
    scale = (absmax / np.float32(127.0)).astype(np.float32)
    q = np.zeros(xf.shape, dtype=np.int8)
    nz = scale > 0
    r = (xf[nz] / scale[nz][:, None]).astype(np.float32)
    q[nz] = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127).astype(np.int8)
    return q, scale


def _int8_quant_scale_128(x):
    xf = oracle.w8a8._as_values(x).astype(np.float32)
    absmax = np.max(np.abs(xf), axis=1)
    scale = (absmax / np.float32(128.0)).astype(np.float32)
    q = np.zeros(xf.shape, dtype=np.int8)
    nz = scale > 0
    q[nz] = np.clip(np.rint(xf[nz] / scale[nz][:, None]), -127, 127).astype(np.int8)
    return q, scale


def _int8_dequant_scales_first(acc, a_scale, b_scale, bias=None):
    f32 = np.float32
    s = (np.asarray(a_scale, dtype=f32)[:, None] * np.asarray(b_scale, dtype=f32)[None, :]).astype(f32)
    v = (np.asarray(acc).astype(f32) * s).astype(f32)
    if bias is not None:
        v = (v + np.asarray(bias, dtype=np.float64).astype(f32)[None, :]).astype(f32)
    return v


def _int8_dequant_no_b_scale(acc, a_scale, b_scale, bias=None):
    return ORIG_INT8_DEQ(acc, a_scale, np.ones_like(np.asarray(b_scale, dtype=np.float32)), bias)


def _int8_dequant_bias_first(acc, a_scale, b_scale, bias=None):
    if bias is None:
        return ORIG_INT8_DEQ(acc, a_scale, b_scale)
    b = np.asarray(bias, dtype=np.float64).astype(np.float32)
    return ORIG_INT8_DEQ(np.asarray(acc).astype(np.float32) + b[None, :], a_scale, b_scale)


def _int8_accumulate_int16(q_a, q_b):
    a = np.asarray(q_a, dtype=np.int8).astype(np.int16)
    b = np.asarray(q_b, dtype=np.int8).astype(np.int16)
    return (a @ b.T).astype(np.int64)


ORIG_F16 = oracle.formats._one_f64_to_f16
ORIG_INT8_DEQ = oracle.w8a8.int8_dequant
ORIG_ACT = oracle.layer.activation
ORIG_DECODE_NVFP4 = oracle.decode.decode_nvfp4
ORIG_LINEAR = oracle.layer.linear

MUTATIONS = {
    "e4m3_bias_8": [(oracle.formats, "_e4m3_value", _e4m3_wrong_bias)],
    "e4m3_flush_subnormals": [(oracle.formats, "_e4m3_value", _e4m3_no_subnormal)],
    "e2m1_sign_in_bit2": [(oracle.formats, "_e2m1_value", _e2m1_sign_bit2)],
    "nvfp4_high_nibble_first": [(oracle.layer, "decode_nvfp4", _nvfp4_high_nibble_first),
                                (oracle, "nvfp4_materialize",
                                 lambda q, bs: _nvfp4_high_nibble_first(q, bs))],
    "nvfp4_block_of_8": [(oracle.layer, "decode_nvfp4", _nvfp4_block_of_8),
                         (oracle, "nvfp4_materialize", _nvfp4_block_of_8)],
    "weight_not_transposed": [(oracle.layer, "linear", _linear_no_transpose)],
    "scale_not_folded": [(oracle.layer, "linear", _linear_drop_alpha)],
    "abs_of_weights": [(oracle.layer, "linear", _linear_abs_weights)],
    "dropped_last_term": [(oracle.layer, "linear", _linear_drop_last_k)],
    "f16_ties_away": [(oracle.formats, "_one_f64_to_f16", _f16_ties_away)],
    "gelu_wrong_cubic": [(oracle.layer, "activation", _gelu_wrong_constant),
                         (oracle, "activation", _gelu_wrong_constant)],
    "silu_wrong_sign": [(oracle.layer, "activation", _silu_wrong_sign),
                        (oracle, "activation", _silu_wrong_sign)],
    "activation_before_bias": [(oracle.layer, "epilogue", _epilogue_act_first),
                               (oracle, "epilogue", _epilogue_act_first)],
    "int8_quant_ties_away": [(oracle, "int8_quantize_rows", _int8_quant_ties_away)],
    "int8_quant_scale_128": [(oracle, "int8_quantize_rows", _int8_quant_scale_128)],
    "int8_dequant_scales_multiplied_first": [
        (oracle.w8a8, "int8_dequant", _int8_dequant_scales_first),
        (oracle, "int8_dequant", _int8_dequant_scales_first)],
    "int8_dequant_no_b_scale": [(oracle.w8a8, "int8_dequant", _int8_dequant_no_b_scale),
                                (oracle, "int8_dequant", _int8_dequant_no_b_scale)],
    "int8_bias_before_dequant": [(oracle.w8a8, "int8_dequant", _int8_dequant_bias_first),
                                 (oracle, "int8_dequant", _int8_dequant_bias_first)],
    "int8_sum_in_int16": [(oracle.w8a8, "int8_accumulate", _int8_accumulate_int16),
                          (oracle, "int8_accumulate", _int8_accumulate_int16)],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    for mod, attr, repl in MUTATIONS[name]:
        monkeypatch.setattr(mod, attr, repl)
    caught = _any_check_fails()
    assert caught is not None, f"no pin catches the planted mistake {name!r}"


def test_grouped_minus_one_not_zeroed_is_caught(monkeypatch):
    orig = oracle.layer.fp8_grouped_matmul

    def leaky(a, w, offs, ids, scales=None, rows=None):
        ids = [0 if int(i) == -1 else int(i) for i in np.asarray(ids).reshape(-1)]
        return orig(a, w, offs, ids, scales, rows)

    monkeypatch.setattr(oracle, "fp8_grouped_matmul", leaky)
    assert _any_check_fails() is not None


def test_unmutated_oracle_passes_every_pin():
    assert _any_check_fails() is None
