// materialize.cu -- dense dequantized copies of the quantized weights.
//
// FP8: out[n, k] = e4m3(w[n, k]); NVFP4: out[n, k] = e2m1(q) * e4m3(bs[n, k/16]).
// Source: the "fp8_gemv" kernel page (enqueue_fp8_materialize /
// fp8_materialize_kernel: the FP8 weight written out as a dense [N, K]
// buffer) and the "fp4_matmul" page for the NVFP4 layout.
//
// Both are flat elementwise maps (input and output share the row-major
// element order), so the kernels walk the flat arrays with a grid-stride loop:
// FP8 in 16-element groups (one 16-byte load), NVFP4 in 16-element blocks
// (8 bytes of nibbles + 1 scale byte).  The conversions are exact, so the
// outputs are bit-exact decodes (HBM-bound: 1 byte in, 2 or 4 bytes out per
// element for FP8).
#include "common.cuh"
#include "internal.h"

namespace gq {
namespace {

constexpr int kThreads = 256;

template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
k_fp8_materialize(void* __restrict__ out, const uint8_t* __restrict__ w, int64_t total) {
  const int64_t groups = total / 16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; g < groups;
       g += stride) {
    const uint4 codes = ld_stream_v4(w + g * 16);
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2(words[i] & 0xFFFFu));
      const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2(words[i] >> 16));
      v[4 * i + 0] = lo.x;
      v[4 * i + 1] = lo.y;
      v[4 * i + 2] = hi.x;
      v[4 * i + 3] = hi.y;
    }
    if constexpr (kBf16) {
      uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + g * 16);
      o[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      o[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                        pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + g * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
  // Tail: the last total % 16 elements, one per thread of block 0.
  if (blockIdx.x == 0) {
    const int64_t t = groups * 16 + threadIdx.x;
    if (t < total) {
      const float v = e4m3_to_f32(w[t]);
      if constexpr (kBf16) {
        static_cast<__nv_bfloat16*>(out)[t] = __float2bfloat16_rn(v);
      } else {
        static_cast<float*>(out)[t] = v;
      }
    }
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
k_nvfp4_materialize(void* __restrict__ out, const uint8_t* __restrict__ q,
                    const uint8_t* __restrict__ bs, int64_t blocks) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; b < blocks;
       b += stride) {
    const uint2 packed = ld_stream_v2(q + b * 8);
    const float scale = e4m3_to_f32(bs[b]);
    const uint32_t words[2] = {packed.x, packed.y};
    float v[16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 e = f16x2_to_f32x2(e2m1x2_to_f16x2(words[i] >> (8 * j)));
        v[8 * i + 2 * j + 0] = e.x * scale;   // exact: <= 6 significant bits
        v[8 * i + 2 * j + 1] = e.y * scale;
      }
    }
    if constexpr (kBf16) {
      uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + b * 16);
      o[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      o[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                        pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + b * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
}

int grid_for(int64_t items, int num_sms) {
  const int64_t want = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 resident CTAs per SM
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_fp8_materialize(const Ctx& c, void* out, bool bf16_out,
                                   const uint8_t* w, int64_t total) {
  const int grid = grid_for(total / 16 > 0 ? total / 16 : 1, c.num_sms);
  if (bf16_out) {
    k_fp8_materialize<true><<<grid, kThreads, 0, c.stream>>>(out, w, total);
  } else {
    k_fp8_materialize<false><<<grid, kThreads, 0, c.stream>>>(out, w, total);
  }
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_materialize(const Ctx& c, void* out, bool bf16_out,
                                     const uint8_t* q, const uint8_t* bs,
                                     int64_t total_blocks) {
  const int grid = grid_for(total_blocks, c.num_sms);
  if (bf16_out) {
    k_nvfp4_materialize<true><<<grid, kThreads, 0, c.stream>>>(out, q, bs, total_blocks);
  } else {
    k_nvfp4_materialize<false><<<grid, kThreads, 0, c.stream>>>(out, q, bs, total_blocks);
  }
  return cudaGetLastError();
}

}  // namespace gq
