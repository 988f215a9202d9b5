"""CPU oracle for the weight-only quantized linear layer  out = x @ dequant(W)^T.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
and reference (``--impl reference``) legs of ``bench.py`` may use it.  It
shares no code with the CUDA library.

It is the plain definition of what the method computes, written out in float64
with numpy:

* the two weight formats decoded through tables built from their bit formulas
  (``formats``): float8_e4m3fn (256 codes) and E2M1 (16 codes);
* the decoded weight (``decode``): FP8 is a table look-up; NVFP4 is the E2M1
  nibble (low nibble first) times the E4M3 block scale of its 16-wide block;
* the linear layer (``linear``): a float64 dot product of the bf16 activations
  with the decoded weight, times the per-tensor scale folded after the sum;
  the grouped (MoE) form loops over groups and runs a dense product per group;
  materialize returns the decoded weight itself;
* the optional fused epilogue (``epilogue``): bias add and an activation,
  and the binary16 output rounding (``formats.f64_to_f16_bits``);
* the W8A8 int8 sibling method (``w8a8``): per-row absmax activation
  quantization, the exact int8 x int8 sum and its float32 dequant.

Sources (Modular kernel API pages for Apple M5):
  * "fp8_gemv" module page: the W8A16 GEMV, the scale contract, materialize;
  * "fp4_matmul" module page: the packed NVFP4 weight layout and block scales;
  * "Matmul2dFp8" struct page, method ``run_grouped``: the grouped MoE product;
    its parameters c_type (fp16 / bf16 / fp32 output) and elementwise_lambda_fn
    (the fused epilogue);
  * "int8_matmul" module page: the W8A8 quantizer and product.

Every function here is pinned by ``tests/test_oracle_pins.py`` against what the
pages and the formats fix (exhaustive code tables, closed forms, brute force in
exact rational arithmetic, invariants).  The pages print no worked numerical
example of the layer itself, so no function is pinned to a printed value.
"""

from .formats import (e4m3_table, e2m1_table, bf16_bits_to_f64, f64_to_bf16_bits,
                      f16_bits_to_f64, f64_to_f16_bits)
from .decode import decode_fp8, decode_nvfp4, nibble
from .w8a8 import (int8_quantize_rows, int8_accumulate, int8_dequant, int8_matmul,
                   int8_abs_sum)
from .layer import (
    linear,
    linear_loops,
    fp8_gemv,
    fp8_matmul,
    nvfp4_gemv,
    nvfp4_matmul,
    fp8_grouped_matmul,
    nvfp4_grouped_matmul,
    fp8_materialize,
    nvfp4_materialize,
    abs_dot,
    bf16_ulp,
    tolerance,
    f16_ulp,
    activation,
    ACT_LIPSCHITZ,
    epilogue,
    tolerance_epilogue,
)

__all__ = [
    "e4m3_table", "e2m1_table", "bf16_bits_to_f64", "f64_to_bf16_bits",
    "decode_fp8", "decode_nvfp4", "nibble",
    "linear", "linear_loops", "fp8_gemv", "fp8_matmul", "nvfp4_gemv",
    "nvfp4_matmul", "fp8_grouped_matmul", "nvfp4_grouped_matmul", "fp8_materialize",
    "nvfp4_materialize", "abs_dot", "bf16_ulp", "tolerance",
    "f16_bits_to_f64", "f64_to_f16_bits", "f16_ulp", "activation", "ACT_LIPSCHITZ",
    "epilogue", "tolerance_epilogue",
    "int8_quantize_rows", "int8_accumulate", "int8_dequant", "int8_matmul", "int8_abs_sum",
]
