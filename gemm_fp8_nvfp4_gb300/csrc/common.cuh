// common.cuh -- device helpers shared by the gq kernels (sm_103a).
//
// Number-format conversions use the hardware cvt instructions, which are
// exact for every code of the narrow formats:
//   float8_e4m3fn pair -> f16x2   (cvt.rn.f16x2.e4m3x2)
//   E2M1 pair (one byte, low nibble = first element) -> f16x2
//                                  (cvt.rn.f16x2.e2m1x2)
// Every E4M3 and E2M1 value (and every E2M1 x E4M3 product) is exact in f16,
// f32 and bf16, so the widenings below never round.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace gq {

// Status bits recorded by bounded waits that ran out (see gq_device_status).
enum : uint32_t {
  kStatusTimeoutProducer = 1u << 0,
  kStatusTimeoutMma = 1u << 1,
  kStatusTimeoutDequant = 1u << 2,
  kStatusTimeoutEpilogue = 1u << 3,
  kStatusTimeoutOther = 1u << 4,
};

// ------------------------------------------------------------------ loads --

// 16-byte streaming load: read once, do not keep in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Cached read-only loads (activations are re-read by many CTAs).
__device__ __forceinline__ uint4 ld_ro_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_ro_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_ro_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// ------------------------------------------------------------ conversions --

// Two float8_e4m3fn codes (low byte = first element) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t out;
  const uint16_t in16 = static_cast<uint16_t>(two_codes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in16));
  return out;
}

// One byte of two E2M1 codes (low nibble = first element) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8) {
  uint32_t out;
  const uint16_t in16 = static_cast<uint16_t>(byte_in_low8 & 0xFFu);
  asm("{\n\t.reg .b8 lo, hi;\n\t"
      "mov.b16 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, lo;\n\t}"
      : "=r"(out)
      : "h"(in16));
  return out;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = h2;
  return __half22float2(h);
}

// bf16x2 bit patterns -> two floats (exact: bf16 is the top half of f32).
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// One float8_e4m3fn code -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  return f16x2_to_f32x2(e4m3x2_to_f16x2(code & 0xFFu)).x;
}

// f16 bits of one float8_e4m3fn code (exact).
__device__ __forceinline__ uint16_t e4m3_to_f16(uint32_t code) {
  return static_cast<uint16_t>(e4m3x2_to_f16x2(code & 0xFFu) & 0xFFFFu);
}

// Both halves of an f16x2 times the f16 s, as two f32: one mixed-precision
// FMA each (fma.rn.f32.f16, f16 inputs, f32 result).  The addend is -0, which
// leaves every product and its sign of zero unchanged; the products used here
// (an E2M1 or E4M3 value times an E4M3 value or 1) have at most 6 significant
// bits, so they are exact.
__device__ __forceinline__ float2 h2_scale_f32(uint32_t h2, uint16_t s) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "fma.rn.f32.f16 %0, l, %3, %4;\n\tfma.rn.f32.f16 %1, h, %3, %4;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2), "h"(s), "f"(-0.0f));
  return make_float2(lo, hi);
}

// Two floats whose low 16 bits are zero (at most 8 significant bits and in the
// bf16 range) -> bf16x2 by taking their high halves: no rounding step.  A NaN
// stays a NaN (the f32 NaNs produced here have a nonzero high mantissa).
__device__ __forceinline__ uint32_t f32x2_hi_to_bf16x2(float2 v) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(r) : "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)));
  return r;
}

// Two e4m3 codes in each half of a 32-bit word -> two f16x2 (hardware cvt,
// exact); the half selection is part of the instruction.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// f16x2 -> (f32, f32).
__device__ __forceinline__ float2 h2f2(uint32_t h) {
  float a, b;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(h));
  return make_float2(a, b);
}

// acc += a * b on both halves: one packed fp32 FMA (fma.rn.f32x2).
__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&acc)));
  acc = *reinterpret_cast<float2*>(&r);
}

// bf16x2 bit patterns -> (f32, f32), exact.
__device__ __forceinline__ float2 bf2f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// Byte B (0..3) of a word holds two E2M1 codes -> f16x2 (hardware cvt, exact).
template <int B>
__device__ __forceinline__ uint32_t e2m1x2_b(uint32_t w) {
  uint32_t out;
  if constexpr (B == 0) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(out) : "r"(w));
  } else if constexpr (B == 1) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}"
        : "=r"(out) : "r"(w));
  } else if constexpr (B == 2) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}"
        : "=r"(out) : "r"(w));
  } else {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}"
        : "=r"(out) : "r"(w));
  }
  return out;
}

// ------------------------------------------------ output and the epilogue --
//
// Every product kernel ends in the same fused epilogue (the optional
// elementwise (row, col) epilogue of the "Matmul2dFp8" struct page, in the
// form a linear layer uses):  out = act(alpha * acc + bias[n]), converted to
// the output type with round-to-nearest-even.

// (Epi and the kOut* / kAct* codes are declared in internal.h.)

__device__ __forceinline__ float epi_bias(const Epi& e, int64_t idx) {
  if (e.bias_kind == kOutF32) return __ldg(static_cast<const float*>(e.bias) + idx);
  const uint16_t b = __ldg(static_cast<const unsigned short*>(e.bias) + idx);
  if (e.bias_kind == kOutBf16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float epi_act(int act, float v) {
  switch (act) {
    case kActRelu: return v > 0.f ? v : (v != v ? v : 0.f);   // NaN stays NaN
    case kActSilu: return v / (1.f + expf(-v));
    case kActGeluTanh:
      return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
    default: return v;
  }
}

// The activation as an out-of-line call: kernels apply the epilogue at many
// unrolled sites, and inlining the transcendental code at each would bloat
// the code that every warp role of a persistent kernel shares.
static __device__ __noinline__ float epi_act_call(int act, float v) { return epi_act(act, v); }

// True when the epilogue is the identity (no bias, no activation): kernels
// test it once per chunk of outputs and skip epi_apply.
__device__ __forceinline__ bool epi_plain(const Epi& e) {
  return e.bias == nullptr && e.act == kActNone;
}

// v = alpha * acc already; adds bias element bias_idx (when there is a bias)
// and applies the activation.
__device__ __forceinline__ float epi_apply(const Epi& e, float v, int64_t bias_idx) {
  if (e.bias != nullptr) v = __fadd_rn(v, epi_bias(e, bias_idx));   // never fused with a product
  if (e.act != kActNone) v = epi_act_call(e.act, v);
  return v;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void epi_store(void* out, int64_t idx, int out_kind, float v) {
  if (out_kind == kOutF32) {
    static_cast<float*>(out)[idx] = v;
  } else if (out_kind == kOutBf16) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

// ----------------------------------------------------------------- stores --

template <typename OutT> struct OutConv;
template <> struct OutConv<float> {
  static __device__ __forceinline__ float cvt(float v) { return v; }
};
template <> struct OutConv<__nv_bfloat16> {
  static __device__ __forceinline__ __nv_bfloat16 cvt(float v) { return __float2bfloat16_rn(v); }
};

// Pack two floats into bf16x2 bits with round-to-nearest-even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four consecutive outputs at idx (idx a multiple of 4, out 16-byte aligned):
// one 16-byte (f32) or 8-byte (bf16, f16) store.
__device__ __forceinline__ void epi_store4(void* out, int64_t idx, int out_kind, float v0, float v1,
                                           float v2, float v3) {
  if (out_kind == kOutF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = make_float4(v0, v1, v2, v3);
  } else if (out_kind == kOutBf16) {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) =
        make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
  } else {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) =
        make_uint2(pack_f16x2(v0, v1), pack_f16x2(v2, v3));
  }
}

// Programmatic dependent launch.  pdl_wait() blocks until the grid this one
// depends on (the previous kernel in the stream, when this kernel was launched
// with programmatic stream serialization) has completed and its memory is
// visible; without such a dependency it returns at once.  Every access to
// memory that the previous kernel may write must come after it.
// pdl_launch_dependents() lets the next kernel start launching early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The same wait without a compiler memory clobber, for kernels whose global
// loads are all volatile asm (never moved across it) and whose stores depend
// on data loaded after it; it keeps register allocation unconstrained.
__device__ __forceinline__ void pdl_wait_ordered() { asm volatile("griddepcontrol.wait;"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t bit) {
  if (status != nullptr) atomicOr(status, bit);
}

}  // namespace gq
