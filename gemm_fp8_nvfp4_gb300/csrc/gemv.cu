// gemv.cu -- M = 1 decode GEMVs for FP8 and NVFP4 weights.
//
//   y[n] = alpha * sum_k x[k] * w_hat[n, k]
//
// Source: the "fp8_gemv" kernel page (fp8_gemv_kernel: the batch-1 decode
// product is a matrix-vector product with no MMA to feed; lanes stride down K
// in vector-wide chunks, widen the FP8 weight to f32 in registers, fp32 FMA,
// warp sum, narrow tail) and, for NVFP4, the same page's description of the
// FP4 sibling (nibble unpack, E2M1 decode, per-16 FP8 block scale) with the
// layout of the "fp4_matmul" page.
//
// GB300 design.  The kernel is HBM-bound: every weight byte is read exactly
// once and nothing else is large.  A CTA of 4 warps owns R = 4 consecutive
// rows and splits K across its 128 threads (thread t takes vectors t, t+128,
// ...), so each thread streams R rows x up to U vectors of 16-byte weight
// loads before it does any arithmetic (deep memory-level parallelism: up to
// 32 KB in flight per CTA), and the bf16 activation chunk it loads once is
// reused for all R rows.  The R partial sums are reduced with xor-shuffles
// inside each warp and then across the 4 warps in a fixed order through
// shared memory (deterministic).
// Weight loads bypass L1 (read once); activation loads go through L1 because
// every CTA on the SM reads the same x.
//
// Every GEMV is launched as a programmatic dependent of the previous kernel
// in the stream (the programmatic stream serialization attribute) and calls
// griddepcontrol.launch_dependents at its start: its CTAs become resident
// while the previous kernel finishes and wait (griddepcontrol.wait) before
// reading or writing global memory, so stream order is kept and the launch
// gap between back-to-back GEMVs is hidden; before that wait they prefetch
// their first weight bytes into L2 (a prefetch returns no data, so what is
// read is unaffected).  With GQ_LAUNCH_OVERLAP_WEIGHT_READS each thread
// issues its first batch of weight loads before that wait, and reads x and
// writes y only after it: the weight stream of one GEMV overlaps the tail of
// the previous kernel -- valid only when that kernel does not write the
// weights, which is why it is opt-in.
//
// The load width adapts to K and the pointers: 16 bytes when K % 16 == 0,
// down to 1 byte for odd K (the pages' scalar tail for K % TILE_K != 0 becomes
// a narrower vector for the whole row, so no row ever straddles an unaligned
// vector).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gq {
namespace {

constexpr int kThreads = 128;   // threads per CTA

// ---------------------------------------------------------------- helpers --

// Weight prefetch before the wait for the previous kernel.  A prefetch
// returns no data, so it may be issued while that kernel still runs: the
// CTA's first weight bytes start moving from HBM into L2 during its tail and
// the loads after the wait find them there.  FP8: the CTA's rows in one
// prefetch when they total at most kPrefetchCtaBytes, else the first
// kPrefetchRowHead bytes of each row: more competes with the loads (whole
// 14 KB rows: 4096 x 14336 took 13.7 us instead of 10.1 us; for the three
// decode shapes back to back with 8-row CTAs at K = 4096, a row head of 2 KB
// or 3 KB ran 3-10 % slower than 1.25 KB, and none at all 9 % slower).
// NVFP4: the CTA's codes and block scales, one prefetch each (at most
// kPrefetchMax).
constexpr int64_t kPrefetchCtaBytes = 16384;
constexpr int64_t kPrefetchRowHead = 1280;
constexpr int64_t kPrefetchMax = 65536;

// L2 prefetch of the 16-byte-aligned part of [p, p + min(bytes, cap)).
__device__ __forceinline__ void prefetch_l2(const uint8_t* p, int64_t bytes, int64_t cap) {
  const uintptr_t a = (reinterpret_cast<uintptr_t>(p) + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t e = (reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(min(bytes, cap))) &
                      ~static_cast<uintptr_t>(15);
  if (e > a) tc::bulk_prefetch_l2(reinterpret_cast<const void*>(a), static_cast<uint32_t>(e - a));
}
// Load VEC bf16 activations starting at element k0 and widen to f32.
template <int VEC>
__device__ __forceinline__ void load_x(const uint16_t* __restrict__ x, int64_t k0, float* xf) {
  if constexpr (VEC == 16) {
    const uint4 a = ld_ro_v4(x + k0);
    const uint4 b = ld_ro_v4(x + k0 + 8);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xf[2 * i] = bf16lo_to_f32(v[i]);
      xf[2 * i + 1] = bf16hi_to_f32(v[i]);
    }
  } else if constexpr (VEC == 8) {
    const uint4 a = ld_ro_v4(x + k0);
    const uint32_t v[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xf[2 * i] = bf16lo_to_f32(v[i]);
      xf[2 * i + 1] = bf16hi_to_f32(v[i]);
    }
  } else if constexpr (VEC == 4) {
    const uint2 a = ld_ro_v2(x + k0);
    xf[0] = bf16lo_to_f32(a.x);
    xf[1] = bf16hi_to_f32(a.x);
    xf[2] = bf16lo_to_f32(a.y);
    xf[3] = bf16hi_to_f32(a.y);
  } else if constexpr (VEC == 2) {
    const uint32_t a = ld_ro_u32(x + k0);
    xf[0] = bf16lo_to_f32(a);
    xf[1] = bf16hi_to_f32(a);
  } else {
    xf[0] = __uint_as_float(static_cast<uint32_t>(x[k0]) << 16);
  }
}

// Load VEC fp8 codes (VEC bytes) of one row as 32-bit words (VEC < 4: one
// word holding the codes in its low bytes).
template <int VEC>
__device__ __forceinline__ void load_w8(const uint8_t* __restrict__ p, uint32_t* words) {
  if constexpr (VEC == 16) {
    const uint4 a = ld_stream_v4(p);
    words[0] = a.x; words[1] = a.y; words[2] = a.z; words[3] = a.w;
  } else if constexpr (VEC == 8) {
    const uint2 a = ld_stream_v2(p);
    words[0] = a.x; words[1] = a.y;
  } else if constexpr (VEC == 4) {
    words[0] = ld_stream_u32(p);
  } else if constexpr (VEC == 2) {
    words[0] = *reinterpret_cast<const uint16_t*>(p);
  } else {
    words[0] = *p;
  }
}

// 16 fp8 codes (4 words) x 16 activations (8 f32 pairs) into a pair
// accumulator: 8 cvt, 8 x 2 cvt.f32.f16 and 8 packed FMAs.
__device__ __forceinline__ void dot16_fp8(const uint32_t* w, const float2* xf, float2& acc) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h01, h23;
    e4m3x4_to_h2x2(w[q], h01, h23);
    ffma2(acc, h2f2(h01), xf[2 * q]);
    ffma2(acc, h2f2(h23), xf[2 * q + 1]);
  }
}

// acc += sum over the VEC codes of x * e4m3(code).
template <int VEC>
__device__ __forceinline__ float fma_fp8(const uint32_t* words, const float* xf, float acc) {
  constexpr int kWords = VEC >= 4 ? VEC / 4 : 1;
#pragma unroll
  for (int i = 0; i < kWords; ++i) {
    if constexpr (VEC >= 2) {
      const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2(words[i] & 0xFFFFu));
      acc = fmaf(xf[4 * i + 0], lo.x, acc);
      acc = fmaf(xf[4 * i + 1], lo.y, acc);
      if constexpr (VEC >= 4) {
        const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2(words[i] >> 16));
        acc = fmaf(xf[4 * i + 2], hi.x, acc);
        acc = fmaf(xf[4 * i + 3], hi.y, acc);
      }
    } else {
      acc = fmaf(xf[0], e4m3_to_f32(words[0]), acc);
    }
  }
  return acc;
}

template <int R, int T>
__device__ __forceinline__ void reduce_and_store(float (&acc)[R], float* red, int64_t row0,
                                                 int64_t N, float alpha, void* y, const Epi& ep) {
  static_assert(R >= 1 && R <= 32 && (R & (R - 1)) == 0, "R must be a power of two <= 32");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Warp sums of the R rows by a transposed butterfly: while n > 1 values are
  // live, the xor step with offset o hands half of them to the partner lane
  // (lanes with bit o set keep the upper half) and adds what comes back, so
  // the first log2(R) steps move n/2 values each instead of R; the remaining
  // steps sum one value.  Lane l then holds the warp's sum of row
  // l / (32 / R), the same in every lane of its group (a fixed order: the
  // result is deterministic).
  float v[R];
#pragma unroll
  for (int r = 0; r < R; ++r) v[r] = acc[r];
#pragma unroll
  for (int off = 16, n = R; off > 0; off >>= 1) {
    if (n > 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
      }
      n >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
    }
  }
  constexpr int kGroup = 32 / R;   // lanes per row after the butterfly
  if (lane % kGroup == 0) red[warp * R + lane / kGroup] = v[0];
  __syncthreads();
  if (threadIdx.x < R) {
    const int r = threadIdx.x;
    float s = 0.f;
#pragma unroll
    for (int wi = 0; wi < T / 32; ++wi) s += red[wi * R + r];
    const int64_t n = row0 + r;
    if (n < N) epi_store(y, n, ep.out_kind, epi_apply(ep, alpha * s, n));
  }
}

// ------------------------------------------------------------------- FP8 --

// kFloor (VEC == 16 only): the same launch, prefetch, wait and weight loads
// with the decode and arithmetic left out -- each thread folds the words it
// loaded into a checksum bit per row -- so its time is the HBM floor of this
// launch shape (gq_probe_gemv_read_floor).
template <int VEC, int R, int U, int T = kThreads, bool kOverlap = false, bool kFloor = false,
          int kMinBlocks = 7>
__global__ void __launch_bounds__(T, kMinBlocks)   // 4 rows: 7 CTAs per SM (<= 73 registers)
k_fp8_gemv(void* __restrict__ y, Epi ep, const uint16_t* __restrict__ x,
           const uint8_t* __restrict__ w, int64_t N, int64_t K, float alpha) {
  constexpr int kThreads = T;
  __shared__ float red[(T / 32) * R];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * R;
  const int64_t nvec = K / VEC;
  // Launched as a programmatic dependent of the previous kernel in the
  // stream: the CTAs become resident while that kernel finishes.  Plain
  // order prefetches the CTA's first weight bytes into L2, then waits for it
  // before reading or writing global memory; overlap mode issues its first
  // batch of weight loads before the wait (x is read and y written only
  // after it).  Every GEMV lets the next kernel's CTAs launch early too: in
  // plain order once its own wait is over (the three decode shapes back to
  // back: 0.4 % faster than at the start of the kernel, where the next
  // kernel's CTAs could take slots before this one's had started).
  if constexpr (!kOverlap || VEC != 16) {
    const int64_t nrows = row0 + R <= N ? R : N - row0;
    if (nrows * K <= kPrefetchCtaBytes) {
      if (threadIdx.x == 0) prefetch_l2(w + row0 * K, nrows * K, kPrefetchCtaBytes);
    } else if (threadIdx.x < nrows) {
      prefetch_l2(w + (row0 + threadIdx.x) * K, K, kPrefetchRowHead);
    }
    pdl_wait();
    pdl_launch_dependents();
  } else {
    pdl_launch_dependents();
  }
  bool waited = !kOverlap || VEC != 16;
  constexpr int kWords = VEC >= 4 ? VEC / 4 : 1;

  // Rows past N (last CTA) re-read the last valid row and are never stored.
  const uint8_t* rows[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t n = row0 + r < N ? row0 + r : N - 1;
    rows[r] = w + n * K;
  }

  float acc[R];
  if constexpr (kFloor) {
    static_assert(VEC == 16, "the read floor follows the 16-byte path");
    uint32_t fold = 0;
    int64_t v = threadIdx.x;
    for (; v + static_cast<int64_t>(U - 1) * kThreads < nvec; v += static_cast<int64_t>(U) * kThreads) {
      uint4 wv[U][R];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < R; ++r) wv[u][r] = ld_stream_v4(rows[r] + (v + u * kThreads) * 16);
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < R; ++r) fold ^= wv[u][r].x ^ wv[u][r].y ^ wv[u][r].z ^ wv[u][r].w;
    }
    for (; v < nvec; v += kThreads) {
      uint4 wv[R];
#pragma unroll
      for (int r = 0; r < R; ++r) wv[r] = ld_stream_v4(rows[r] + v * 16);
#pragma unroll
      for (int r = 0; r < R; ++r) fold ^= wv[r].x ^ wv[r].y ^ wv[r].z ^ wv[r].w;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = static_cast<float>((fold >> r) & 1u);
  } else if constexpr (VEC == 16) {
    // 16 codes per vector; the activations are widened once per vector and
    // reused for the R rows; pair accumulators fed by packed FMAs.
    float2 acc2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc2[r] = make_float2(0.f, 0.f);
    int64_t v = threadIdx.x;
    for (; v + static_cast<int64_t>(U - 1) * kThreads < nvec; v += static_cast<int64_t>(U) * kThreads) {
      uint4 wv[U][R];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < R; ++r) wv[u][r] = ld_stream_v4(rows[r] + (v + u * kThreads) * 16);
      if (!waited) {
        pdl_wait_ordered();
        waited = true;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint4 xa = ld_ro_v4(x + (v + u * kThreads) * 16);
        const uint4 xb = ld_ro_v4(x + (v + u * kThreads) * 16 + 8);
        const float2 xf[8] = {bf2f2(xa.x), bf2f2(xa.y), bf2f2(xa.z), bf2f2(xa.w),
                              bf2f2(xb.x), bf2f2(xb.y), bf2f2(xb.z), bf2f2(xb.w)};
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t ww[4] = {wv[u][r].x, wv[u][r].y, wv[u][r].z, wv[u][r].w};
          dot16_fp8(ww, xf, acc2[r]);
        }
      }
    }
    for (; v < nvec; v += kThreads) {
      uint4 wv[R];
#pragma unroll
      for (int r = 0; r < R; ++r) wv[r] = ld_stream_v4(rows[r] + v * 16);
      if (!waited) {
        pdl_wait_ordered();
        waited = true;
      }
      const uint4 xa = ld_ro_v4(x + v * 16);
      const uint4 xb = ld_ro_v4(x + v * 16 + 8);
      const float2 xf[8] = {bf2f2(xa.x), bf2f2(xa.y), bf2f2(xa.z), bf2f2(xa.w),
                            bf2f2(xb.x), bf2f2(xb.y), bf2f2(xb.z), bf2f2(xb.w)};
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t ww[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
        dot16_fp8(ww, xf, acc2[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = acc2[r].x + acc2[r].y;
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    int64_t v = threadIdx.x;
    for (; v + static_cast<int64_t>(U - 1) * kThreads < nvec; v += static_cast<int64_t>(U) * kThreads) {
      uint32_t wv[U][R][kWords];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < R; ++r) load_w8<VEC>(rows[r] + (v + u * kThreads) * VEC, wv[u][r]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float xf[VEC];
        load_x<VEC>(x, (v + u * kThreads) * VEC, xf);
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = fma_fp8<VEC>(wv[u][r], xf, acc[r]);
      }
    }
    for (; v < nvec; v += kThreads) {
      uint32_t wv[R][kWords];
#pragma unroll
      for (int r = 0; r < R; ++r) load_w8<VEC>(rows[r] + v * VEC, wv[r]);
      float xf[VEC];
      load_x<VEC>(x, v * VEC, xf);
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = fma_fp8<VEC>(wv[r], xf, acc[r]);
    }
  }
  if (!waited) pdl_wait_ordered();   // threads without a vector still order their store
  reduce_and_store<R, T>(acc, red, row0, N, alpha, y, ep);
}

// ----------------------------------------------------------------- NVFP4 --

// One vector = VB bytes of packed nibbles = 2*VB elements = VB/8 blocks; xf
// holds the vector's activations as f32 pairs (VB pairs).
template <int VB>
__device__ __forceinline__ void dot_nvfp4(const uint32_t* words, uint32_t scales, const float2* xf,
                                          float2& acc) {
  constexpr int kBlocks = VB / 8;
#pragma unroll
  for (int b = 0; b < kBlocks; ++b) {
    float2 part = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t wd = words[2 * b + q];
      ffma2(part, h2f2(e2m1x2_b<0>(wd)), xf[8 * b + 4 * q + 0]);
      ffma2(part, h2f2(e2m1x2_b<1>(wd)), xf[8 * b + 4 * q + 1]);
      ffma2(part, h2f2(e2m1x2_b<2>(wd)), xf[8 * b + 4 * q + 2]);
      ffma2(part, h2f2(e2m1x2_b<3>(wd)), xf[8 * b + 4 * q + 3]);
    }
    const float s = e4m3_to_f32(scales >> (8 * b));
    ffma2(acc, part, make_float2(s, s));
  }
}

template <int VB>
__device__ __forceinline__ void load_xf(const uint16_t* __restrict__ x, int64_t k0, float2* xf) {
#pragma unroll
  for (int q = 0; q < VB / 4; ++q) {
    const uint4 xv = ld_ro_v4(x + k0 + 8 * q);
    xf[4 * q + 0] = bf2f2(xv.x);
    xf[4 * q + 1] = bf2f2(xv.y);
    xf[4 * q + 2] = bf2f2(xv.z);
    xf[4 * q + 3] = bf2f2(xv.w);
  }
}

// kFloor: weight and scale loads only (as in k_fp8_gemv).
template <int VB, int R, int U, int T = kThreads, bool kOverlap = false, bool kFloor = false>
__global__ void __launch_bounds__(T, 7)   // 7 CTAs per SM (<= 73 registers)
k_nvfp4_gemv(void* __restrict__ y, Epi ep, const uint16_t* __restrict__ x,
             const uint8_t* __restrict__ q, const uint8_t* __restrict__ bs, int64_t N,
             int64_t K, float alpha) {
  constexpr int kThreads = T;
  __shared__ float red[(T / 32) * R];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * R;
  const int64_t half_k = K / 2;
  // Programmatic dependent launch as in k_fp8_gemv.
  pdl_launch_dependents();
  if constexpr (!kOverlap) {
    if (threadIdx.x == 0) {
      const int64_t nrows = row0 + R <= N ? R : N - row0;
      prefetch_l2(q + row0 * half_k, nrows * half_k, kPrefetchMax);
      prefetch_l2(bs + row0 * (K / 16), nrows * (K / 16), kPrefetchMax);
    }
    pdl_wait();
  }
  bool waited = !kOverlap;
  const int64_t nvec = half_k / VB;
  constexpr int kWords = VB / 4;
  constexpr int kBlocks = VB / 8;
  float2 acc2[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc2[r] = make_float2(0.f, 0.f);
  const uint8_t* qrows[R];
  const uint8_t* srows[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t n = row0 + r < N ? row0 + r : N - 1;
    qrows[r] = q + n * half_k;
    srows[r] = bs + n * (K / 16);
  }
  auto load_scales = [&](const uint8_t* s, int64_t vv) -> uint32_t {
    if constexpr (kBlocks == 2) {
      return *reinterpret_cast<const uint16_t*>(s + vv * 2);
    } else {
      return s[vv];
    }
  };

  uint32_t fold = 0;   // kFloor: checksum of the loaded words
  int64_t v = threadIdx.x;
  for (; v + static_cast<int64_t>(U - 1) * kThreads < nvec; v += static_cast<int64_t>(U) * kThreads) {
    uint32_t wv[U][R][kWords];
    uint32_t sv[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        load_w8<VB>(qrows[r] + (v + u * kThreads) * VB, wv[u][r]);
        sv[u][r] = load_scales(srows[r], v + u * kThreads);
      }
    if (!waited) {
      pdl_wait_ordered();
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if constexpr (kFloor) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int i = 0; i < kWords; ++i) fold ^= wv[u][r][i] ^ sv[u][r];
      } else {
        float2 xf[VB];
        load_xf<VB>(x, (v + u * kThreads) * 2 * VB, xf);
#pragma unroll
        for (int r = 0; r < R; ++r) dot_nvfp4<VB>(wv[u][r], sv[u][r], xf, acc2[r]);
      }
    }
  }
  for (; v < nvec; v += kThreads) {
    uint32_t wv[R][kWords];
    uint32_t sv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      load_w8<VB>(qrows[r] + v * VB, wv[r]);
      sv[r] = load_scales(srows[r], v);
    }
    if (!waited) {
      pdl_wait_ordered();
      waited = true;
    }
    if constexpr (kFloor) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < kWords; ++i) fold ^= wv[r][i] ^ sv[r];
    } else {
      float2 xf[VB];
      load_xf<VB>(x, v * 2 * VB, xf);
#pragma unroll
      for (int r = 0; r < R; ++r) dot_nvfp4<VB>(wv[r], sv[r], xf, acc2[r]);
    }
  }
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    acc[r] = kFloor ? static_cast<float>((fold >> r) & 1u) : acc2[r].x + acc2[r].y;
  if (!waited) pdl_wait_ordered();   // threads without a vector still order their store
  reduce_and_store<R, T>(acc, red, row0, N, alpha, y, ep);
}

constexpr int kRows = 4;

// MINB: CTAs per SM the register budget allows; MINB_OV: the same for the
// overlap-mode instantiation (which keeps more values live across the wait).
template <int VEC, int R, int U, int MINB = 7, int MINB_OV = MINB>
cudaError_t fp8_launch(const Ctx& c, void* y, const Epi& ep, const void* x,
                       const uint8_t* w, int64_t N, int64_t K, float alpha) {
  const int64_t grid = (N + R - 1) / R;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (c.overlap_weights) {
    return launch_kernel(c, true, k_fp8_gemv<VEC, R, U, kThreads, true, false, MINB_OV>,
                         dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, y, ep,
                         static_cast<const uint16_t*>(x), w, N, K, alpha);
  }
  return launch_kernel(c, true, k_fp8_gemv<VEC, R, U, kThreads, false, false, MINB>,
                       dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, y, ep,
                       static_cast<const uint16_t*>(x), w, N, K, alpha);
}

// Launch shape of the 16-byte-vector FP8 GEMV (also used by its read-floor
// probe).  A thread with exactly two vectors per row (K = 4096) issues all
// of its rows' vectors in one batch (U = 2: one memory round trip instead of
// two), in 8-row CTAs (96 registers: at most 5 per SM) whose free slots let
// the next kernel of the stream start its prologue and L2 prefetch while
// this one drains; alone, 4096 x 4096 takes 4.5-4.8 us instead of 3.5 us and
// 14336 x 4096 11.3 us instead of 11.0 us with 4-row CTAs, but the three
// decode shapes in sequence take 26.1 us instead of 26.7 us (4-row CTAs for
// 14336 x 4096; at most 4 8-row CTAs per SM: 26.3 us; measured back to back
// on one GPU).  Otherwise (K = 14336) 4-row CTAs take a batch of four
// vectors, then single ones.
enum class Fp8Shape { kR4U4, kR8U2 };
Fp8Shape fp8_shape(const Ctx&, int64_t, int64_t K) {
  return (K / 16 + kThreads - 1) / kThreads == 2 ? Fp8Shape::kR8U2 : Fp8Shape::kR4U4;
}

template <int VEC>
cudaError_t fp8_dispatch(const Ctx& c, void* y, const Epi& ep, const void* x,
                         const uint8_t* w, int64_t N, int64_t K, float alpha) {
  if constexpr (VEC == 16) {
    switch (fp8_shape(c, N, K)) {
      case Fp8Shape::kR8U2: return fp8_launch<16, 8, 2, 5, 4>(c, y, ep, x, w, N, K, alpha);
      default: return fp8_launch<16, kRows, 4>(c, y, ep, x, w, N, K, alpha);
    }
  }
  return fp8_launch<VEC, kRows, 2>(c, y, ep, x, w, N, K, alpha);
}

}  // namespace

cudaError_t launch_gemv_read_floor(const Ctx& c, int format, void* y, const uint8_t* w,
                                   const uint8_t* bs, int64_t N, int64_t K) {
  const int64_t grid = (N + kRows - 1) / kRows;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  Epi ep{};
  ep.out_kind = kOutBf16;
  const dim3 g(static_cast<unsigned>(grid));
  if (format == 0) {
    const auto* none = static_cast<const uint16_t*>(nullptr);
    switch (fp8_shape(c, N, K)) {
      case Fp8Shape::kR8U2:
        return launch_kernel(c, true, k_fp8_gemv<16, 8, 2, kThreads, false, true, 5>,
                             dim3(static_cast<unsigned>((N + 7) / 8)), dim3(kThreads), 0, y, ep, none,
                             w, N, K, 1.0f);
      default:
        return launch_kernel(c, true, k_fp8_gemv<16, kRows, 4, kThreads, false, true>, g,
                             dim3(kThreads), 0, y, ep, none, w, N, K, 1.0f);
    }
  }
  return launch_kernel(c, true, k_nvfp4_gemv<8, kRows, 2, kThreads, false, true>, g, dim3(kThreads), 0,
                       y, ep, static_cast<const uint16_t*>(nullptr), w, bs, N, K, 1.0f);
}

cudaError_t launch_fp8_gemv(const Ctx& c, void* y, const Epi& ep, const void* x,
                            const uint8_t* w, int64_t N, int64_t K, float alpha) {
  const uintptr_t wa = reinterpret_cast<uintptr_t>(w);
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
  auto fits = [&](int vec) {
    return K % vec == 0 && wa % vec == 0 && xa % (vec >= 8 ? 16 : 2 * vec) == 0;
  };
  if (fits(16)) return fp8_dispatch<16>(c, y, ep, x, w, N, K, alpha);
  if (fits(8)) return fp8_dispatch<8>(c, y, ep, x, w, N, K, alpha);
  if (fits(4)) return fp8_dispatch<4>(c, y, ep, x, w, N, K, alpha);
  if (fits(2)) return fp8_dispatch<2>(c, y, ep, x, w, N, K, alpha);
  return fp8_dispatch<1>(c, y, ep, x, w, N, K, alpha);
}

cudaError_t launch_nvfp4_gemv(const Ctx& c, void* y, const Epi& ep, const void* x,
                              const uint8_t* q, const uint8_t* bs, int64_t N,
                              int64_t K, float alpha) {
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  // 4 rows per CTA, two 8-byte vectors (one 16-element block each) per row
  // per step: measured best at N = K = 4096 against 16-byte vectors and
  // other row / vector / CTA-size splits.  At most 7 CTAs per SM (72
  // registers) put the 1024 CTAs of N = 4096 in one wave (1064 slots); with 6
  // per SM, 112 CTAs ran as a second wave (3.91 us against 3.56 us; 8 per SM
  // 4.12 us, 8-row CTAs 3.89 us).
  const int64_t grid = (N + kRows - 1) / kRows;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (c.overlap_weights) {
    return launch_kernel(c, true, k_nvfp4_gemv<8, kRows, 2, kThreads, true>,
                         dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, y, ep, xb, q,
                         bs, N, K, alpha);
  }
  return launch_kernel(c, true, k_nvfp4_gemv<8, kRows, 2>,
                       dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, y, ep, xb, q,
                       bs, N, K, alpha);
}

}  // namespace gq
