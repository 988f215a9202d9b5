// gemm_common.cuh -- pieces shared by the two tcgen05 GEMM kernels (gemm.cu,
// gemm_skinny.cu): the exact weight decode into bf16 shared-memory tiles and
// the host-side tensor-map encoders.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace gq {

// ------------------------------------------------------------- dequant --

// The decodes below run on the dequant warps' critical path, so they keep the
// float conversions to one per pair of elements: the hardware cvt to f16x2,
// then a mixed-precision FMA to f32 (exact), then the bf16 is the f32's high
// half (exact: every value has at most 6 significant bits).

// 16 FP8 codes -> 16 bf16 (two 16-byte chunks), exact, NaN preserved.
__device__ __forceinline__ void fp8x16_to_bf16(uint4 v, uint4& lo, uint4& hi) {
  constexpr uint16_t kOne = 0x3C00;   // 1.0 in f16
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h01, h23;
    e4m3x4_to_h2x2(w[i], h01, h23);
    o[2 * i] = f32x2_hi_to_bf16x2(h2_scale_f32(h01, kOne));
    o[2 * i + 1] = f32x2_hi_to_bf16x2(h2_scale_f32(h23, kOne));
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// 16 int8 codes -> 16 binary16, exactly: each byte's sign bit is flipped
// (u = code + 128, 0..255), the byte becomes the low byte of the binary16
// 0x6400 | u = 1024 + u (spacing 1 in [1024, 2048)), and 1152 is subtracted
// (exact: the result is the integer code in [-128, 127]).
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t u, uint32_t sel) {
  uint32_t h, d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(h) : "r"(u), "r"(0x64646464u), "r"(sel));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(0x64806480u));
  return d;
}

__device__ __forceinline__ void s8x16_to_f16(uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;
    o[2 * i] = s8x2_to_f16x2(u, 0x5140u);       // codes 4i, 4i+1
    o[2 * i + 1] = s8x2_to_f16x2(u, 0x5342u);   // codes 4i+2, 4i+3
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// 8 packed bytes (16 E2M1 codes, low nibble first) x one E4M3 block scale
// (given as f16 bits) -> 16 bf16, exact (the product has at most 6
// significant bits and lies in [2^-10, 2688]).
__device__ __forceinline__ void nvfp4x16_to_bf16(uint32_t w0, uint32_t w1, uint16_t scale_h,
                                                 uint4& lo, uint4& hi) {
  uint32_t o[8];
  o[0] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<0>(w0), scale_h));
  o[1] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<1>(w0), scale_h));
  o[2] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<2>(w0), scale_h));
  o[3] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<3>(w0), scale_h));
  o[4] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<0>(w1), scale_h));
  o[5] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<1>(w1), scale_h));
  o[6] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<2>(w1), scale_h));
  o[7] = f32x2_hi_to_bf16x2(h2_scale_f32(e2m1x2_b<3>(w1), scale_h));
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Byte offset of the 16-byte chunk `j` of row `r` in a K-major tile stored
// with the 128-byte swizzle (rows of 128 bytes, 8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t sw128_off(int r, int j) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

// ----------------------------------------------------------- tensor maps --

// Encoders for the driver's cuTensorMapEncodeTiled (resolved at run time).
inline bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                      uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle sw) {
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0, d0 * d1};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gq
