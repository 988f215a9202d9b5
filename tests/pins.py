"""Checks that pin the CPU oracle to facts fixed outside the oracle itself.

Each ``check_*`` returns None when the oracle passes and raises AssertionError
otherwise.  ``test_oracle_pins.py`` runs them on the oracle as it is;
``test_oracle_mutations.py`` plants plausible mistakes in the oracle and shows
that at least one check fails for each.

What the checks compare against (never the oracle's own formulas):
* hand-worked golden fixtures under ``tests/golden/`` (code tables, a worked
  FP8 GEMV, a worked NVFP4 GEMV, a worked grouped product);
* torch's own float8_e4m3fn -> float32 and float32 -> bfloat16 conversions
  (library routines: the special cases of the decode and the rounding);
* exact rational arithmetic (``fractions.Fraction``) on tiny shapes, with the
  weight decoded independently (torch for E4M3, the golden table for E2M1,
  nibbles and block scales indexed element by element);
* invariants the method states: the scale fold is exact, the GEMV is the M = 1
  row of the GEMM, grouped equals per-group dense products, -1 writes zeros;
* for the W8A8 int8 method: a hand-worked example, and scalar re-statements
  in plain Python (integer sums; float32 rounding through ``struct``) of the
  quantizer and the dequant.
"""

from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- fixtures --

def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def _num(tok: str) -> float:
    return float("nan") if tok == "nan" else float(tok)


def golden_e2m1() -> dict:
    return {int(c): _num(v) for c, v in _lines("e2m1_codes.txt")}


def golden_e4m3() -> dict:
    return {int(c, 16): _num(v) for c, v in _lines("e4m3_landmarks.txt")}


def _rows(name):
    out = {}
    for tok in _lines(name):
        out.setdefault(tok[0], []).append(tok[1:])
    return out


def _same(a: float, b: float) -> bool:
    """Equal as values, NaN matches NaN, and the sign of zero matters."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


# ------------------------------------------------- independent decode paths --

def torch_e4m3(codes) -> np.ndarray:
    """E4M3 codes -> float64 through torch's float8_e4m3fn type."""
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def fraction_of(v: float) -> Fraction:
    return Fraction(v)  # exact for any finite binary float


def exact_fp8_linear(x_vals, w_codes, alpha):
    """Exact alpha * x @ W^T with W decoded through torch, as Fractions."""
    w = torch_e4m3(w_codes)
    m_rows, k_len = x_vals.shape
    n_rows = w.shape[0]
    out = [[None] * n_rows for _ in range(m_rows)]
    for m in range(m_rows):
        for n in range(n_rows):
            s = Fraction(0)
            for k in range(k_len):
                s += fraction_of(float(x_vals[m, k])) * fraction_of(float(w[n, k]))
            out[m][n] = fraction_of(alpha) * s
    return out


def exact_nvfp4_linear(x_vals, q, bs, alpha):
    """Exact product with the NVFP4 weight decoded element by element:
    element k of row n is nibble (k % 2) of byte k // 2 (low nibble first)
    times the E4M3 value of block scale k // 16."""
    t4 = golden_e2m1()
    scale_vals = torch_e4m3(bs)
    m_rows, k_len = x_vals.shape
    n_rows = q.shape[0]
    out = [[None] * n_rows for _ in range(m_rows)]
    for m in range(m_rows):
        for n in range(n_rows):
            s = Fraction(0)
            for k in range(k_len):
                byte = int(q[n, k // 2])
                code = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
                w = fraction_of(t4[code]) * fraction_of(float(scale_vals[n, k // 16]))
                s += fraction_of(float(x_vals[m, k])) * w
            out[m][n] = fraction_of(alpha) * s
    return out


def _bf16_values(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    return bits, x.to(torch.float64).numpy()


# ------------------------------------------------------------------- checks --

def check_e4m3_table(orc):
    t8 = orc.e4m3_table()
    assert t8.shape == (256,)
    for code, val in golden_e4m3().items():
        assert _same(float(t8[code]), val), (hex(code), t8[code], val)
    nan_codes = [c for c in range(256) if math.isnan(t8[c])]
    assert nan_codes == [0x7F, 0xFF], nan_codes
    finite = t8[~np.isnan(t8)]
    assert finite.size == 254
    assert finite.max() == 448.0 and finite.min() == -448.0
    pos = t8[0x00:0x7F]
    assert np.all(np.diff(pos) > 0), "E4M3 codes 0x00..0x7E must increase"
    for c in range(0x80):
        a, b = t8[c], t8[c | 0x80]
        assert _same(float(b), -float(a)) or (math.isnan(a) and math.isnan(b))
    lib = torch_e4m3(np.arange(256))
    for c in range(256):
        assert _same(float(t8[c]), float(lib[c])), hex(c)


def check_e2m1_table(orc):
    t4 = orc.e2m1_table()
    gold = golden_e2m1()
    assert t4.shape == (16,)
    for code, val in gold.items():
        assert _same(float(t4[code]), val), (code, t4[code], val)


def _sig_bits(v: float) -> int:
    """Number of significant bits of a finite dyadic value."""
    if v == 0:
        return 0
    fr = Fraction(abs(v))
    num, den = fr.numerator, fr.denominator
    while num % 2 == 0:
        num //= 2
    return num.bit_length()


def check_bf16_exactness(orc):
    """Every E2M1 * E4M3 product (and every E4M3 value) is exact in bf16:
    at most 8 significant bits and inside the normal bf16 range; torch's
    float64 -> bf16 cast returns it unchanged."""
    t4, t8 = orc.e2m1_table(), orc.e4m3_table()
    prods = []
    for a in t4:
        for b in t8:
            if math.isnan(b):
                continue
            prods.append(float(a) * float(b))
    prods += [float(b) for b in t8 if not math.isnan(b)]
    arr = np.array(prods)
    for v in prods:
        assert _sig_bits(v) <= 6, v
        assert v == 0 or 2.0 ** -126 <= abs(v) < 2.0 ** 128
    back = torch.from_numpy(arr).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(back, arr)
    bits = orc.f64_to_bf16_bits(arr)
    assert np.array_equal(orc.bf16_bits_to_f64(bits), arr)


def check_bf16_rounding(orc):
    """The oracle's float64 -> bf16 rounding equals torch's float32 -> bf16
    cast (round to nearest even) on float32-representable inputs, including
    ties, subnormals, overflow and signed zero."""
    rng = np.random.default_rng(7)
    vals = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    raw = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    rand_bits = raw.view(np.float32)
    rand_bits = rand_bits[np.isfinite(rand_bits)]
    ties = (np.arange(1, 200, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    special = np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.4e38, -3.4e38,
                        1e-40, -1e-40, 1.1754944e-38, 9.2e-41], dtype=np.float32)
    allv = np.concatenate([vals, rand_bits, ties.view(np.float32), special])
    lib = torch.from_numpy(allv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = orc.f64_to_bf16_bits(allv.astype(np.float64))
    assert np.array_equal(mine, lib), np.nonzero(mine != lib)[0][:5]


def check_bf16_decode(orc):
    rng = np.random.default_rng(3)
    bits, vals = _bf16_values(rng, (500,))
    assert np.array_equal(orc.bf16_bits_to_f64(bits), vals)


def check_fp8_worked(orc):
    rows = _rows("fp8_gemv_worked.txt")
    x = np.array([float(v) for v in rows["x"][0]])
    w = np.array([[int(c, 16) for c in r] for r in rows["w"]], dtype=np.uint8)
    alpha = float(rows["alpha"][0][0])
    raw = [float(v) for v in rows["raw"][0]]
    scaled = [float(v) for v in rows["scaled"][0]]
    got_raw = orc.fp8_gemv(x, w, 1.0)
    got_scaled = orc.fp8_gemv(x, w, alpha)
    assert np.array_equal(got_raw, raw), got_raw
    assert np.array_equal(got_scaled, scaled), got_scaled
    assert np.array_equal(orc.linear_loops(x, orc.decode_fp8(w), alpha)[0], scaled)


def check_nvfp4_worked(orc):
    rows = _rows("nvfp4_gemv_worked.txt")
    q = np.array([[int(c, 16) for c in rows["q"][0]]], dtype=np.uint8)
    bs = np.array([[int(c, 16) for c in rows["bs"][0]]], dtype=np.uint8)
    x = np.array([float(v) for v in rows["x"][0]])
    alpha = float(rows["alpha"][0][0])
    raw = float(rows["raw"][0][0])
    scaled = float(rows["scaled"][0][0])
    assert orc.nvfp4_gemv(x, q, bs, 1.0)[0] == raw
    assert orc.nvfp4_gemv(x, q, bs, alpha)[0] == scaled
    assert orc.nvfp4_matmul(x[None, :], q, bs, alpha)[0, 0] == scaled


def check_grouped_worked(orc):
    rows = _rows("grouped_worked.txt")
    w = np.zeros((2, 2, 2), dtype=np.uint8)
    w[0] = [[int(c, 16) for c in r] for r in rows["w0"]]
    w[1] = [[int(c, 16) for c in r] for r in rows["w1"]]
    scales = np.array([float(v) for v in rows["scales"][0]])
    offs = np.array([int(v) for v in rows["a_offsets"][0]])
    ids = np.array([int(v) for v in rows["expert_ids"][0]])
    a = np.array([[float(v) for v in r] for r in rows["a"]])
    want = np.array([[float(v) for v in r] for r in rows["out"]])
    got, written = orc.fp8_grouped_matmul(a, w, offs, ids, scales)
    assert written.all()
    assert np.array_equal(got, want), got
    # the -1 group's rows are exactly zero
    assert np.all(got[2:4] == 0.0)


def _close_to_exact(got: float, exact: Fraction, terms_abs: Fraction, k_len: int):
    """float64 sum of k exact products vs the exact sum: within k * 2^-52 of
    the absolute sum (the float64 summation bound)."""
    err = abs(Fraction(got) - exact)
    return err <= Fraction(k_len + 1, 2 ** 52) * terms_abs


def check_bruteforce_fp8(orc, seed=11, trials=6):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        m, n, k = int(rng.integers(1, 5)), int(rng.integers(1, 5)), int(rng.integers(1, 49))
        bits, xv = _bf16_values(rng, (m, k))
        w = rng.integers(0, 256, size=(n, k), dtype=np.uint8)
        w[(w & 0x7F) == 0x7F] = 0x3C          # keep NaN codes out of sums
        alpha = float(rng.choice([1.0, 0.5, 0.0731]))
        exact = exact_fp8_linear(xv, w, alpha)
        absw = np.abs(torch_e4m3(w))
        got = orc.fp8_matmul(bits, w, alpha)
        got_loops = orc.linear_loops(bits, orc.decode_fp8(w), alpha)
        assert got.shape == (m, n)
        for i in range(m):
            for j in range(n):
                tabs = abs(Fraction(alpha)) * sum(
                    Fraction(abs(float(xv[i, kk]))) * Fraction(float(absw[j, kk])) for kk in range(k))
                assert _close_to_exact(float(got[i, j]), exact[i][j], tabs, k), (t, i, j)
                assert _close_to_exact(float(got_loops[i, j]), exact[i][j], tabs, k), (t, i, j)


def check_bruteforce_nvfp4(orc, seed=12, trials=5):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        m, n = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        k = 16 * int(rng.integers(1, 4))
        bits, xv = _bf16_values(rng, (m, k))
        q = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
        bs = rng.integers(0, 0x7F, size=(n, k // 16), dtype=np.uint8)
        alpha = float(rng.choice([1.0, 0.25, 0.013]))
        exact = exact_nvfp4_linear(xv, q, bs, alpha)
        got = orc.nvfp4_matmul(bits, q, bs, alpha)
        assert got.shape == (m, n)
        wabs = np.abs(orc.decode_nvfp4(q, bs))
        for i in range(m):
            for j in range(n):
                tabs = abs(Fraction(alpha)) * sum(
                    Fraction(abs(float(xv[i, kk]))) * Fraction(float(wabs[j, kk])) for kk in range(k))
                assert _close_to_exact(float(got[i, j]), exact[i][j], tabs, k), (t, i, j)


def check_nvfp4_materialize_independent(orc, seed=13):
    """Materialize equals the element-by-element decode (nibble k % 2 of byte
    k // 2 times block scale k // 16), exactly, signs of zero included."""
    rng = np.random.default_rng(seed)
    n, k = 3, 64
    q = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    bs = rng.integers(0, 256, size=(n, k // 16), dtype=np.uint8)
    t4 = golden_e2m1()
    sv = torch_e4m3(bs)
    got = orc.nvfp4_materialize(q, bs)
    for r in range(n):
        for c in range(k):
            byte = int(q[r, c // 2])
            code = (byte & 0xF) if c % 2 == 0 else (byte >> 4)
            want = t4[code] * float(sv[r, c // 16])
            assert _same(float(got[r, c]), want), (r, c)


def check_fp8_materialize_independent(orc):
    codes = np.arange(256, dtype=np.uint8).reshape(2, 128)
    got = orc.fp8_materialize(codes)
    lib = torch_e4m3(codes)
    for idx in np.ndindex(codes.shape):
        assert _same(float(got[idx]), float(lib[idx]))


def check_scale_fold(orc, seed=14):
    """A power-of-two per-tensor scale factors out of the float64 sum exactly
    (the fold after the product is exact, as the FP8 page states)."""
    rng = np.random.default_rng(seed)
    bits, _ = _bf16_values(rng, (3, 40))
    w = rng.integers(0, 0x7F, size=(5, 40), dtype=np.uint8)
    raw = orc.fp8_matmul(bits, w, 1.0)
    for alpha in (0.5, 2.0 ** -7, 8.0):
        assert np.array_equal(orc.fp8_matmul(bits, w, alpha), alpha * raw)
    q = rng.integers(0, 256, size=(4, 16), dtype=np.uint8)
    bs = rng.integers(0, 0x7F, size=(4, 2), dtype=np.uint8)
    raw4 = orc.nvfp4_matmul(bits[:, :32], q, bs, 1.0)
    assert np.array_equal(orc.nvfp4_matmul(bits[:, :32], q, bs, 0.25), 0.25 * raw4)


def check_gemv_is_gemm_row(orc, seed=15):
    rng = np.random.default_rng(seed)
    bits, xv = _bf16_values(rng, (4, 32))
    w = rng.integers(0, 0x7F, size=(6, 32), dtype=np.uint8)
    g = orc.linear_loops(bits, orc.decode_fp8(w), 0.75)
    for i in range(4):
        v = orc.linear_loops(bits[i], orc.decode_fp8(w), 0.75)[0]
        assert np.array_equal(v, g[i])
        assert np.allclose(orc.fp8_gemv(bits[i], w, 0.75), g[i], rtol=1e-13, atol=0)
    q = rng.integers(0, 256, size=(6, 16), dtype=np.uint8)
    bs = rng.integers(0, 0x7F, size=(6, 2), dtype=np.uint8)
    gm = orc.nvfp4_matmul(bits[:, :32], q, bs, 0.5)
    for i in range(4):
        assert np.allclose(orc.nvfp4_gemv(bits[i, :32], q, bs, 0.5), gm[i], rtol=1e-13, atol=0)


def check_grouped_vs_dense(orc, seed=16):
    """Grouped equals a dense product per group; -1 and unknown ids give zeros;
    empty groups and rows outside every group are untouched."""
    rng = np.random.default_rng(seed)
    e, n, k = 3, 5, 32
    w = rng.integers(0, 0x7F, size=(e, n, k), dtype=np.uint8)
    scales = np.array([0.5, 2.0, 0.125])
    offs = np.array([1, 4, 4, 9, 12, 15])        # row 0 and rows >= 15 uncovered
    ids = np.array([2, 0, -1, 1, 7])              # 7 is outside [0, E): zeros
    bits, _ = _bf16_values(rng, (17, k))
    got, written = orc.fp8_grouped_matmul(bits, w, offs, ids, scales)
    assert not written[0] and not written[15] and not written[16]
    assert np.all(np.isnan(got[0])) and np.all(np.isnan(got[15:]))
    t8 = torch_e4m3(w.reshape(-1)).reshape(w.shape)
    xv = orc.bf16_bits_to_f64(bits)
    for z, ex in enumerate(ids):
        r0, r1 = offs[z], offs[z + 1]
        for r in range(r0, r1):
            if ex == -1 or not (0 <= ex < e):
                assert np.all(got[r] == 0.0)
            else:
                want = scales[ex] * (t8[ex] @ xv[r])
                assert np.allclose(got[r], want, rtol=1e-12, atol=0)
    # rows= sampling returns the same values for the chosen rows
    sub, _ = orc.fp8_grouped_matmul(bits, w, offs, ids, scales, rows=[2, 10, 13])
    for r in (2, 10, 13):
        assert np.array_equal(sub[r], got[r])


def check_tolerance_shape(orc):
    """The tolerance is 2e-4 * |alpha| * sum |x w|; bf16 adds one ulp."""
    x = np.array([[1.0, -2.0]])
    w = np.array([[3.0, 4.0]])
    tol = orc.tolerance(x, w, -0.5)
    assert tol.shape == (1, 1) and tol[0, 0] == 2e-4 * 0.5 * 11.0
    tb = orc.tolerance(x, w, 1.0, out_bf16=True)
    # ref = -5; |ref| + tol in [4, 8): bf16 ulp 2^-5
    assert tb[0, 0] == 2e-4 * 11.0 + 2.0 ** -5


def check_f16_decode(orc):
    """Every binary16 pattern decodes to numpy's float16 value (a library
    special case of the same format), NaN exactly at the NaN patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_bits_to_f64(bits)
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    m = ~np.isnan(want)
    assert np.array_equal(got[m], want[m])
    assert np.array_equal(np.signbit(got[m]), np.signbit(want[m]))
    assert got[0x7BFF] == 65504.0 and got[0x0001] == 2.0 ** -24 and got[0x7C00] == np.inf


def check_f16_rounding(orc, seed=21):
    """float64 -> binary16 RNE agrees with numpy's conversion on values at
    every scale, on exact ties between neighbours (both parities), around
    the overflow threshold and in the subnormal range."""
    rng = np.random.default_rng(seed)
    vals = [rng.standard_normal(400) * 10.0 ** rng.integers(-9, 6, 400)]
    halves = orc.f16_bits_to_f64(np.arange(0, 0x7C00, 97, dtype=np.uint32).astype(np.uint16))
    nxt = orc.f16_bits_to_f64(np.arange(1, 0x7C01, 97, dtype=np.uint32).astype(np.uint16))
    vals.append((halves + nxt) / 2.0)                      # exact midpoints (ties)
    vals.append(np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e6, 2.0 ** -25, 3 * 2.0 ** -26,
                          2.0 ** -24 * 1.5, -0.0, 0.0, np.inf, -np.inf]))
    v = np.concatenate(vals)
    v = np.concatenate([v, -v])
    got = orc.f64_to_f16_bits(v)
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    assert orc.f64_to_f16_bits(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


def check_activations(orc):
    """Activations against what their definitions fix: ReLU's closed form;
    the odd parts of SiLU and tanh-GELU are v / 2 (act(v) - act(-v) = v);
    slope 1/2 at 0; SiLU's sigmoid limits; tanh-GELU within the approximation's
    known distance (< 1e-3) of the erf form 0.5 v (1 + erf(v / sqrt 2));
    the Lipschitz bounds the tolerance uses are tight upper bounds."""
    v = np.linspace(-8.0, 8.0, 3201)
    r = orc.activation(v, "relu")
    assert np.array_equal(r, np.where(v > 0, v, 0.0))
    assert np.isnan(orc.activation(np.array([np.nan]), "relu")[0])
    assert np.array_equal(orc.activation(v, "none"), v)
    for kind in ("silu", "gelu_tanh"):
        a = orc.activation(v, kind)
        assert np.allclose(a - orc.activation(-v, kind), v, rtol=1e-12, atol=1e-12)
        h = 1e-6
        d0 = (orc.activation(np.array([h]), kind) - orc.activation(np.array([-h]), kind))[0] / (2 * h)
        assert abs(d0 - 0.5) < 1e-6
        slope = np.max(np.abs(np.diff(a) / np.diff(v)))
        assert orc.ACT_LIPSCHITZ[kind] - 0.02 < slope <= orc.ACT_LIPSCHITZ[kind]
    s = orc.activation(np.array([40.0, -40.0, 0.0]), "silu")
    assert abs(s[0] - 40.0) < 1e-12 and abs(s[1]) < 1e-15 and s[2] == 0.0
    g = orc.activation(v, "gelu_tanh")
    erf_form = np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in v])
    assert np.max(np.abs(g - erf_form)) < 1e-3


def check_epilogue(orc):
    """The bias is added per output column before the activation."""
    v = np.array([[1.0, -1.0], [0.5, 4.0]])
    b = np.array([-2.0, 3.0])
    out = orc.epilogue(v, b, "relu")
    assert np.array_equal(out, np.array([[0.0, 2.0], [0.0, 7.0]]))
    assert np.array_equal(orc.epilogue(v, None, "none"), v)
    # tolerance: Lipschitz bound x pre-activation tolerance + 2^-20 |out| (+ output ulp)
    t = orc.tolerance_epilogue(np.array([1e-3]), np.array([3.0]), "silu", "f32")
    assert t[0] == 1.1 * 1e-3 + 3.0 * 2.0 ** -20
    t16 = orc.tolerance_epilogue(np.array([0.0]), np.array([3.0]), "none", "f16")
    assert t16[0] == 3.0 * 2.0 ** -20 + 2.0 ** -9      # f16 ulp on [2, 4) is 2^-9


def check_nvfp4_grouped_worked(orc):
    rows = _rows("nvfp4_grouped_worked.txt")
    q = np.zeros((2, 2, 8), dtype=np.uint8)
    bs = np.zeros((2, 2, 1), dtype=np.uint8)
    for e in range(2):
        q[e] = [[int(c, 16) for c in r] for r in rows[f"q{e}"]]
        bs[e] = [[int(c, 16) for c in r] for r in rows[f"bs{e}"]]
    scales = np.array([float(v) for v in rows["scales"][0]])
    offs = np.array([int(v) for v in rows["a_offsets"][0]])
    ids = np.array([int(v) for v in rows["expert_ids"][0]])
    a = np.array([[float(v) for v in r] for r in rows["a"]])
    want = np.array([[float(v) for v in r] for r in rows["out"]])
    got, written = orc.nvfp4_grouped_matmul(a, q, bs, offs, ids, scales)
    assert written.all()
    assert np.array_equal(got, want), got


def check_nvfp4_grouped_vs_dense(orc, seed=17):
    """NVFP4 grouped equals, row by row, the second scale times the product
    with an independent element-by-element decode of the expert's weight;
    -1 and unknown ids give zeros, uncovered rows stay unwritten."""
    rng = np.random.default_rng(seed)
    e, n, k = 3, 4, 32
    q = rng.integers(0, 256, size=(e, n, k // 2), dtype=np.uint8)
    bs = rng.integers(0, 0x7F, size=(e, n, k // 16), dtype=np.uint8)
    scales = np.array([0.25, 2.0, 1.5])
    offs = np.array([1, 3, 3, 6, 8])
    ids = np.array([2, 0, -1, 5])
    bits, _ = _bf16_values(rng, (9, k))
    got, written = orc.nvfp4_grouped_matmul(bits, q, bs, offs, ids, scales)
    assert not written[0] and not written[8]
    t4 = golden_e2m1()
    xv = orc.bf16_bits_to_f64(bits)
    for z, ex in enumerate(ids):
        for r in range(offs[z], offs[z + 1]):
            if ex == -1 or not (0 <= ex < e):
                assert np.all(got[r] == 0.0)
                continue
            sv = torch_e4m3(bs[ex])
            for col in range(n):
                acc = 0.0
                for c in range(k):
                    byte = int(q[ex, col, c // 2])
                    code = (byte & 0xF) if c % 2 == 0 else (byte >> 4)
                    acc += xv[r, c] * t4[code] * float(sv[col, c // 16])
                assert np.isclose(got[r, col], scales[ex] * acc, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- W8A8 int8 --

def _f32(v: float) -> float:
    """Round a Python float (binary64) to the nearest binary32 (ties to even)."""
    return struct.unpack("<f", struct.pack("<f", v))[0]


def check_int8_worked(orc):
    rows = _rows("int8_w8a8_worked.txt")
    x = np.array([[float(v) for v in r] for r in rows["x"]])
    want_q = np.array([[int(v) for v in r] for r in rows["q"]], dtype=np.int8)
    absmax = [float(v) for v in rows["absmax"][0]]
    q, scale = orc.int8_quantize_rows(x)
    assert np.array_equal(q, want_q), q
    for i, am in enumerate(absmax):
        assert scale[i] == np.float32(_f32(am / 127.0)), (i, scale[i])
    assert scale[1] == 1.0 and scale[2] == 0.0
    b = np.array([[int(v) for v in r] for r in rows["b"]], dtype=np.int8)
    acc = orc.int8_accumulate(q, b)
    want_acc = np.array([[int(v) for v in r] for r in rows["acc"]])
    assert np.array_equal(acc, want_acc), acc
    b_scale = np.array([float(v) for v in rows["b_scale"][0]], dtype=np.float32)
    bias = np.array([float(v) for v in rows["bias"][0]])
    out = orc.int8_matmul(q, b, scale, b_scale, bias).astype(np.float64)
    want = np.array([[float(v) for v in r] for r in rows["out"]])
    assert np.array_equal(out[1:], want[1:]), out
    assert np.allclose(out[0], want[0], rtol=4 * 2.0 ** -24, atol=0), out


def check_int8_quantizer_scalar(orc, seed=31):
    """The quantizer equals a plain-Python restatement: absmax, scale =
    absmax / 127 and x / scale each rounded once to binary32 (a binary64
    result rounded to binary32 is the correctly rounded binary32 result for
    a quotient of binary32 values), Python's round (half to even), clamp."""
    rng = np.random.default_rng(seed)
    bits, _ = _bf16_values(rng, (6, 40))
    # a row whose absmax is 127 (scale 1) with exact halves, and a zero row
    xv = orc.bf16_bits_to_f64(bits)
    xv[4] = 0.0
    xv[5, :8] = [127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -126.5]
    xv[5, 8:] = np.round(xv[5, 8:] * 8) / 8
    q, scale = orc.int8_quantize_rows(xv)
    for i in range(xv.shape[0]):
        am = max(abs(float(v)) for v in xv[i])
        s = _f32(am / 127.0)
        assert float(scale[i]) == s, (i, scale[i], s)
        for j in range(xv.shape[1]):
            if s == 0.0:
                want = 0
            else:
                want = max(-127, min(127, round(_f32(float(xv[i, j]) / s))))
            assert int(q[i, j]) == want, (i, j, int(q[i, j]), want)


def check_int8_quantizer_invariants(orc, seed=32):
    """|q| <= 127; the absmax element gets +-127; x - q * scale is at most half
    a step; q(-x) = -q(x)."""
    rng = np.random.default_rng(seed)
    bits, _ = _bf16_values(rng, (5, 64))
    xv = orc.bf16_bits_to_f64(bits)
    q, scale = orc.int8_quantize_rows(xv)
    qn, scale_n = orc.int8_quantize_rows(-xv)
    assert np.array_equal(scale, scale_n) and np.array_equal(qn, -q)
    assert np.all(np.abs(q.astype(np.int64)) <= 127)
    for i in range(xv.shape[0]):
        j = int(np.argmax(np.abs(xv[i])))
        assert abs(int(q[i, j])) == 127
        err = np.abs(xv[i] - q[i].astype(np.float64) * float(scale[i]))
        assert np.all(err <= 0.5 * float(scale[i]) * (1 + 2.0 ** -20)), err.max()


def check_int8_product_scalar(orc, seed=33):
    """The exact sums equal Python integer loops; the dequant equals the
    float32 steps (acc * a_scale) * b_scale + bias done one by one through
    ``struct``; sums beyond 2^24 (K = 1100, all codes +-127) round once."""
    rng = np.random.default_rng(seed)
    m, n, k = 8, 16, 9
    qa = rng.integers(-127, 128, size=(m, k), dtype=np.int8)
    qb = rng.integers(-127, 128, size=(n, k), dtype=np.int8)
    sa = (rng.random(m) * 0.02).astype(np.float32)
    sb = (rng.random(n) * 0.01).astype(np.float32)
    bias = np.round(rng.standard_normal(n) * 8) / 8
    acc = orc.int8_accumulate(qa, qb)
    out = orc.int8_dequant(acc, sa, sb, bias)
    for i in range(m):
        for j in range(n):
            s = sum(int(qa[i, c]) * int(qb[j, c]) for c in range(k))
            assert int(acc[i, j]) == s
            v = _f32(_f32(_f32(float(s)) * float(sa[i])) * float(sb[j]))
            v = _f32(v + float(bias[j]))
            assert float(out[i, j]) == v, (i, j, float(out[i, j]), v)
    big_a = np.full((1, 1100), 127, dtype=np.int8)
    big_b = np.full((1, 1100), -127, dtype=np.int8)
    big_b[0, 0] = 126
    s = 126 * 127 - 1099 * 127 * 127
    assert int(orc.int8_accumulate(big_a, big_b)[0, 0]) == s
    assert float(orc.int8_dequant(np.array([[s]]), [1.0], [1.0])[0, 0]) == _f32(float(s))


ALL_CHECKS = [
    check_e4m3_table, check_e2m1_table, check_bf16_exactness, check_bf16_rounding,
    check_bf16_decode, check_fp8_worked, check_nvfp4_worked, check_grouped_worked,
    check_bruteforce_fp8, check_bruteforce_nvfp4, check_nvfp4_materialize_independent,
    check_fp8_materialize_independent, check_scale_fold, check_gemv_is_gemm_row,
    check_grouped_vs_dense, check_tolerance_shape, check_f16_decode, check_f16_rounding,
    check_activations, check_epilogue, check_nvfp4_grouped_worked, check_nvfp4_grouped_vs_dense,
    check_int8_worked, check_int8_quantizer_scalar, check_int8_quantizer_invariants,
    check_int8_product_scalar,
]
