"""Weight decode (dequant) for the two formats, float64.

Test infrastructure only (see the package docstring).

FP8 ("fp8_gemv" module page, the paragraph on the FP8 sibling of the FP4
GEMV): the weight is float8_e4m3fn [N, K], one byte per element, and the
decoded weight is the code's value.

NVFP4 ("fp4_matmul" module page, first paragraph): the weight stays packed as
uint8 [N, K/2] with the low nibble first plus float8_e4m3fn block scales
[N, K/16].  Element k of row n is the E2M1 code in nibble (k mod 2) of byte
k // 2 -- the low nibble holds the even element -- and its value is that E2M1
value times the E4M3 value of the scale of its 16-wide block, bs[n, k // 16].
"""

import numpy as np

from .formats import e2m1_table, e4m3_table


def nibble(byte: int, which: int) -> int:
    """Nibble ``which`` (0 = low, holds the even element; 1 = high) of a byte."""
    return (byte & 0xF) if which == 0 else (byte >> 4) & 0xF


def decode_fp8(w_codes) -> np.ndarray:
    """uint8 [..., K] float8_e4m3fn codes -> float64 [..., K]."""
    t8 = e4m3_table()
    return t8[np.asarray(w_codes, dtype=np.uint8)]


def decode_nvfp4(q_packed, block_scales) -> np.ndarray:
    """Packed NVFP4 weight -> float64 [N, K].

    q_packed:     uint8 [N, K/2]; byte j of a row holds element 2j in its low
                  nibble and element 2j+1 in its high nibble.
    block_scales: uint8 [N, K/16] float8_e4m3fn codes, one per 16 consecutive
                  elements of a row.
    """
    q = np.asarray(q_packed, dtype=np.uint8)
    bs = np.asarray(block_scales, dtype=np.uint8)
    n_rows, half_k = q.shape
    k = 2 * half_k
    if k % 16 != 0:
        raise ValueError("NVFP4 needs K to be a multiple of the 16-element block")
    if bs.shape != (n_rows, k // 16):
        raise ValueError("block scales must be [N, K/16]")
    t4 = e2m1_table()
    t8 = e4m3_table()
    codes = np.empty((n_rows, k), dtype=np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    scale_per_element = np.repeat(t8[bs], 16, axis=1)
    return t4[codes] * scale_per_element
