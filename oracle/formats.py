"""Number formats used by the layer, decoded from their bit formulas (float64).

Test infrastructure only (see the package docstring).

* float8_e4m3fn -- the FP8 weight of the "fp8_gemv" module page and the block
  scale of the NVFP4 weight on the "fp4_matmul" module page.  One sign bit,
  four exponent bits (bias 7), three mantissa bits; the ``fn`` variant has no
  infinities, the all-ones exponent with all-ones mantissa is NaN, so the
  largest finite magnitude is 1.75 * 2^8 = 448.  Exponent field 0 encodes the
  subnormals m/8 * 2^-6.  The pages require the decode to be exact for every
  code (the "fp8_gemv" page, the paragraph on the denormal flush-to-zero
  hazard), so the table is exact rational arithmetic carried in float64.
* E2M1 -- the 4-bit weight element of the "fp4_matmul" page.  One sign bit
  (bit 3), two exponent bits (bias 1), one mantissa bit; exponent field 0 is
  the subnormal m * 0.5.  Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* bfloat16 -- the activation type: the top 16 bits of an IEEE binary32.
* binary16 (fp16) -- an output type (the "Matmul2dFp8" struct page lists fp16,
  bf16 and fp32 for c_type): one sign bit, five exponent bits (bias 15), ten
  mantissa bits; exponent field 0 encodes the subnormals m/1024 * 2^-14.
"""

import math

import numpy as np


def _e4m3_value(code: int) -> float:
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def _e2m1_value(code: int) -> float:
    s = (code >> 3) & 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = m * 0.5
    else:
        mag = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def e4m3_table() -> np.ndarray:
    """float64[256]: value of every float8_e4m3fn code (NaN for 0x7F, 0xFF)."""
    return np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e2m1_table() -> np.ndarray:
    """float64[16]: value of every E2M1 code (code 8 is -0.0)."""
    return np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64 values (exact).

    A bfloat16 is the upper half of a binary32, so the value is the binary32
    whose high 16 bits are the pattern and whose low 16 bits are zero.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    """float64 -> bfloat16 bit patterns with round-to-nearest-even.

    Written from the definition: find the two bf16 neighbours of the float64
    value (8 significant bits) and pick the nearer one, the one with an even
    last bit on a tie.  Overflow past the largest bf16 gives +-inf, NaN stays
    NaN (quiet, 0x7FC0 with the input's sign), subnormals are kept.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_in = v.reshape(-1)
    flat_out = out.reshape(-1)
    for i, x in enumerate(flat_in):
        flat_out[i] = _one_f64_to_bf16(float(x))
    return out


def _one_f64_to_bf16(x: float) -> int:
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    if math.isnan(x):
        return sign | 0x7FC0
    a = abs(x)
    if math.isinf(a):
        return sign | 0x7F80
    if a == 0.0:
        return sign
    # bf16: 8 exponent bits (bias 127), 7 stored mantissa bits.
    # The quantum (ulp) for normal values in [2^e, 2^(e+1)) is 2^(e-7);
    # for subnormals (below 2^-126) it is 2^-133.
    m, e = math.frexp(a)          # a = m * 2^e, m in [0.5, 1)
    e2 = e - 1                    # a in [2^e2, 2^(e2+1))
    q_exp = max(e2, -126) - 7
    scaled = math.ldexp(a, -q_exp)  # exact (power-of-two scaling)
    n = math.floor(scaled)
    frac = scaled - n
    if frac > 0.5 or (frac == 0.5 and (n & 1)):
        n += 1
    r = math.ldexp(n, q_exp)      # rounded magnitude, exact
    if r >= 2.0 ** 128:
        return sign | 0x7F80
    # Re-encode r as bf16 bits.
    if r < 2.0 ** -126:
        mant = int(math.ldexp(r, 133))        # subnormal: r = mant * 2^-133
        return sign | mant
    m2, e3 = math.frexp(r)
    exp_field = (e3 - 1) + 127
    mant = int(math.ldexp(m2, 8)) - 128       # 7 stored bits
    return sign | (exp_field << 7) | mant


def f16_bits_to_f64(bits) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> float64, decoded from the fields."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = (b & 0x3FF).astype(np.float64)
    normal = sign * (1.0 + m / 1024.0) * np.ldexp(1.0, (e - 15))
    sub = sign * (m / 1024.0) * 2.0 ** -14
    special = np.where(m == 0, sign * np.inf, np.nan)
    return np.where(e == 0x1F, special, np.where(e == 0, sub, normal))


def f64_to_f16_bits(v) -> np.ndarray:
    """float64 -> binary16 bit patterns with round-to-nearest-even.

    Same construction as the bfloat16 rounding: the value's quantum is
    2^(e-10) for magnitudes in [2^e, 2^(e+1)) and 2^-24 below 2^-14 (the
    subnormals); round to a multiple of it, ties to the even multiple; a
    rounded magnitude of 2^16 or more is infinity (largest finite 65504).
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_in = v.reshape(-1)
    flat_out = out.reshape(-1)
    for i, x in enumerate(flat_in):
        flat_out[i] = _one_f64_to_f16(float(x))
    return out


def _one_f64_to_f16(x: float) -> int:
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    if math.isnan(x):
        return sign | 0x7E00
    a = abs(x)
    if math.isinf(a):
        return sign | 0x7C00
    if a == 0.0:
        return sign
    m, e = math.frexp(a)
    e2 = e - 1
    q_exp = max(e2, -14) - 10
    scaled = math.ldexp(a, -q_exp)
    n = math.floor(scaled)
    frac = scaled - n
    if frac > 0.5 or (frac == 0.5 and (n & 1)):
        n += 1
    r = math.ldexp(n, q_exp)
    if r >= 2.0 ** 16:
        return sign | 0x7C00
    if r < 2.0 ** -14:
        return sign | int(math.ldexp(r, 24))          # subnormal: r = mant * 2^-24
    m2, e3 = math.frexp(r)
    exp_field = (e3 - 1) + 15
    mant = int(math.ldexp(m2, 11)) - 1024             # 10 stored bits
    return sign | (exp_field << 10) | mant
