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

// 16 consecutive values at element idx (16 * sizeof(out type) bytes,
// 16-byte aligned): float32, bfloat16 or binary16 (all exact here).
template <int kOut>
__device__ __forceinline__ void store16(void* out, int64_t idx, const float (&v)[16]) {
  if constexpr (kOut == kOutF32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = kOut == kOutBf16 ? pack_bf16x2(v[2 * i], v[2 * i + 1]) : pack_f16x2(v[2 * i], v[2 * i + 1]);
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx);
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int kOut>
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
    store16<kOut>(out, g * 16, v);
  }
  // Tail: the last total % 16 elements, one per thread of block 0.
  if (blockIdx.x == 0) {
    const int64_t t = groups * 16 + threadIdx.x;
    if (t < total) {
      epi_store(out, t, kOut, e4m3_to_f32(w[t]));
    }
  }
}

template <int kOut>
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
    store16<kOut>(out, b * 16, v);
  }
}

int grid_for(int64_t items, int num_sms) {
  const int64_t want = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 resident CTAs per SM
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_fp8_materialize(const Ctx& c, void* out, int out_kind,
                                   const uint8_t* w, int64_t total) {
  const int grid = grid_for(total / 16 > 0 ? total / 16 : 1, c.num_sms);
  if (out_kind == kOutBf16) k_fp8_materialize<kOutBf16><<<grid, kThreads, 0, c.stream>>>(out, w, total);
  else if (out_kind == kOutF16) k_fp8_materialize<kOutF16><<<grid, kThreads, 0, c.stream>>>(out, w, total);
  else k_fp8_materialize<kOutF32><<<grid, kThreads, 0, c.stream>>>(out, w, total);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_materialize(const Ctx& c, void* out, int out_kind,
                                     const uint8_t* q, const uint8_t* bs,
                                     int64_t total_blocks) {
  const int grid = grid_for(total_blocks, c.num_sms);
  if (out_kind == kOutBf16)
    k_nvfp4_materialize<kOutBf16><<<grid, kThreads, 0, c.stream>>>(out, q, bs, total_blocks);
  else if (out_kind == kOutF16)
    k_nvfp4_materialize<kOutF16><<<grid, kThreads, 0, c.stream>>>(out, q, bs, total_blocks);
  else
    k_nvfp4_materialize<kOutF32><<<grid, kThreads, 0, c.stream>>>(out, q, bs, total_blocks);
  return cudaGetLastError();
}

}  // namespace gq
