// fewrow.cu -- W8A16 / W4A16 products with at most 16 activation rows on
// register-fed tensor-core MMAs.
//
//   C[m, n] = alpha * sum_k A[m, k] * w_hat[n, k]      (A bf16, fp32 accumulate)
//
// Source: the "fp8_gemv" page (decode-sized products are weight-read bound:
// the weight streams once, is widened in registers and multiplied with the
// few activation rows) and the "fp4_matmul" page (NVFP4 layout: packed E2M1
// codes, low nibble first, one E4M3 block scale per 16 elements).
//
// GB300 design.  With M <= 16 every weight element is read, decoded and used
// once, by at most 16 activation rows: the tensor-core work is tiny, and a
// tcgen05 tile would pad M to 128 and serialise K/16 MMAs of ~150 cycles per
// CTA.  Here the weights stream like the GEMV's and feed the warp-level MMA
// mma.sync.m16n8k16 (bf16 x bf16 -> f32) straight from registers:
//   * one CTA per SM, 16 warps, takes an even contiguous share of the N
//     weight rows and walks it in groups of 32 rows (two 16-row MMA tiles;
//     rows past the share are zero and never loaded); its warps take the K
//     steps w, w + 16, ..., issuing the weight loads of two steps before
//     the decode and MMAs of the first;
//   * in a K step, lane (g, t) (g = lane / 4, t = lane % 4) loads the 16-byte
//     chunk t of rows g and g + 8 of each tile (FP8: 16 elements, NVFP4: 32
//     elements = two blocks and their two scale bytes) and decodes it exactly
//     to bf16 in registers;
//   * MMA j of the chunk takes elements 4j .. 4j + 3 of every lane's chunk:
//     MMA column slots 2t, 2t + 1 hold elements 4j, 4j + 1 and slots 2t + 8,
//     2t + 9 hold 4j + 2, 4j + 3, so the k a slot stands for depends only on
//     (t, j), the same for all 16 rows, and the activation fragment of token
//     n is the 4 consecutive activations at k = step + t * chunk + 4j;
//   * activations (bf16, read-only, shared by every CTA) come through L1;
//     tokens 0..7 form the first 8-column MMA tile, tokens 8..15 the second
//     (skipped for M <= 8); tokens >= M are zero columns;
//   * the 16 warps' partial tiles are summed in a fixed order in shared
//     memory, then alpha, the fused epilogue and the output conversion.
// Launched as a programmatic dependent of the previous kernel (like the
// GEMVs): set-up and an L2 prefetch of the CTA's weight rows overlap that
// kernel's tail; every read of A or the weights and every write follow
// griddepcontrol.wait.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <algorithm>

namespace gq {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTiles = 2;                 // 16-row MMA tiles per row group
constexpr int kGroupRows = 16 * kTiles;   // weight rows per row group
constexpr int kMaxM = 16;                 // activation rows (two 8-column MMA tiles)
constexpr int kFewFp8 = 0, kFewNvfp4 = 1;
constexpr int kBatch = 2;                // K steps whose weight loads are issued together

// D (16 x 8, f32) += A (16 x 16, bf16, row-major fragment) x B (16 x 8, bf16).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8 bf16 activations of one token starting at k (16-byte aligned), or zeros.
__device__ __forceinline__ uint4 act8(const uint16_t* __restrict__ a, bool ok, int64_t off) {
  return ok ? ld_ro_v4(a + off) : make_uint4(0u, 0u, 0u, 0u);
}

// 16-byte weight chunk (and, NVFP4, the two block scales under it) of one
// row, or zeros for a row outside the CTA's range.
template <int F>
__device__ __forceinline__ void load_chunk(const uint8_t* __restrict__ w, const uint8_t* __restrict__ bs,
                                           bool ok, int64_t row, int64_t rbytes, int64_t K,
                                           int64_t k0, uint4& v, uint32_t& sc) {
  if (!ok) {
    v = make_uint4(0u, 0u, 0u, 0u);
    sc = 0u;
    return;
  }
  v = ld_stream_v4(w + row * rbytes + (F == kFewFp8 ? k0 : k0 / 2));
  if constexpr (F == kFewNvfp4) sc = *reinterpret_cast<const uint16_t*>(bs + row * (K / 16) + k0 / 16);
  else sc = 0u;
}

// The chunk of one row as bf16 words (word i = elements 2i, 2i + 1), exact.
template <int F>
__device__ __forceinline__ void decode_chunk(uint4 v, uint32_t sc, uint32_t (&o)[F == kFewFp8 ? 8 : 16]) {
  uint4 p, q;
  if constexpr (F == kFewFp8) {
    fp8x16_to_bf16(v, p, q);
    o[0] = p.x; o[1] = p.y; o[2] = p.z; o[3] = p.w; o[4] = q.x; o[5] = q.y; o[6] = q.z; o[7] = q.w;
  } else {
    nvfp4x16_to_bf16(v.x, v.y, e4m3_to_f16(sc), p, q);
    o[0] = p.x; o[1] = p.y; o[2] = p.z; o[3] = p.w; o[4] = q.x; o[5] = q.y; o[6] = q.z; o[7] = q.w;
    nvfp4x16_to_bf16(v.z, v.w, e4m3_to_f16(sc >> 8), p, q);
    o[8] = p.x; o[9] = p.y; o[10] = p.z; o[11] = p.w; o[12] = q.x; o[13] = q.y; o[14] = q.z; o[15] = q.w;
  }
}

template <int F, bool kTwo>
__global__ void __launch_bounds__(kThreads, 1)
k_fewrow(void* __restrict__ out, Epi ep, const uint16_t* __restrict__ a,
         const uint8_t* __restrict__ w, const uint8_t* __restrict__ bs, int M, int64_t N,
         int64_t K, float alpha) {
  constexpr int kChunk = F == kFewFp8 ? 16 : 32;      // elements per 16-byte chunk
  constexpr int kStepK = 4 * kChunk;                  // K per warp step (4 lanes per row)
  constexpr int kJ = kChunk / 4;                      // MMAs per chunk and tile
  constexpr int kWords = kChunk / 2;
  __shared__ float red[kWarps][kGroupRows][kMaxM];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // This CTA's rows: an even share of N (contiguous), in groups of kGroupRows.
  const int64_t r_begin = static_cast<int64_t>(blockIdx.x) * N / gridDim.x;
  const int64_t r_end = static_cast<int64_t>(blockIdx.x + 1) * N / gridDim.x;
  const int64_t rbytes = F == kFewFp8 ? K : K / 2;     // weight bytes per row
  pdl_launch_dependents();
  // L2 prefetch of each row before the wait (a prefetch returns no data).
  // FP8: the whole row (up to 64 KB).  NVFP4: the first 1 KB of the codes and
  // the row's block scales -- at M = 16 and N = K = 4096 7.54 us against
  // 7.70 us with the whole codes and no scales (M = 8: 5.78 / 5.93 us).
  constexpr int64_t kHead = F == kFewFp8 ? 65536 : 1024;
  for (int64_t r = r_begin + threadIdx.x; r < r_end; r += kThreads) {
    tc::bulk_prefetch_l2_span(w + r * rbytes, rbytes < kHead ? rbytes : kHead);
    if constexpr (F == kFewNvfp4) tc::bulk_prefetch_l2_span(bs + r * (K / 16), K / 16 < 65536 ? K / 16 : 65536);
  }
  pdl_wait();

  const bool tok0 = g < M, tok1 = kTwo && g + 8 < M;
  const uint16_t* a0 = a + static_cast<int64_t>(tok0 ? g : 0) * K;
  const uint16_t* a1 = a + static_cast<int64_t>(tok1 ? g + 8 : 0) * K;
  const int64_t nsteps = K / kStepK;

  for (int64_t row0 = r_begin; row0 < r_end; row0 += kGroupRows) {
    // lane rows: tile i holds rows row0 + 16 i + g and row0 + 16 i + g + 8
    int64_t rows[kTiles][2];
    bool ok[kTiles][2];
#pragma unroll
    for (int i = 0; i < kTiles; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        rows[i][h] = row0 + 16 * i + g + 8 * h;
        ok[i][h] = rows[i][h] < r_end;
      }
    float d[kTiles][2][4];
#pragma unroll
    for (int i = 0; i < kTiles; ++i)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[i][c][e] = 0.f;

    for (int64_t s0 = warp; s0 < nsteps; s0 += static_cast<int64_t>(kWarps) * kBatch) {
      // The weight chunks (and NVFP4 block scales) of kBatch steps first, so
      // one memory round trip serves them; then per step the activation
      // fragments (k0 .. k0 + chunk of each token: L1 / L2 hits), the decode
      // and the MMAs.
      uint4 wv[kBatch][kTiles][2];
      uint32_t sv[kBatch][kTiles][2];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int64_t s = s0 + static_cast<int64_t>(kWarps) * b;
        const int64_t k0 = s * kStepK + t * kChunk;
#pragma unroll
        for (int i = 0; i < kTiles; ++i)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            load_chunk<F>(w, bs, ok[i][h] && s < nsteps, rows[i][h], rbytes, K, k0, wv[b][i][h],
                          sv[b][i][h]);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int64_t s = s0 + static_cast<int64_t>(kWarps) * b;
        if (s >= nsteps) break;
        const int64_t k0 = s * kStepK + t * kChunk;
        uint4 x0[kJ / 2], x1[kJ / 2];
#pragma unroll
        for (int jj = 0; jj < kJ / 2; ++jj) {
          x0[jj] = act8(a0, tok0, k0 + 8 * jj);
          x1[jj] = kTwo ? act8(a1, tok1, k0 + 8 * jj) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kTiles; ++i) {
          uint32_t lo[kWords], hi[kWords];
          decode_chunk<F>(wv[b][i][0], sv[b][i][0], lo);
          decode_chunk<F>(wv[b][i][1], sv[b][i][1], hi);
#pragma unroll
          for (int j = 0; j < kJ; ++j) {
            // activations k0 + 4j .. k0 + 4j + 3: word pair (2 (j % 2), + 1) of x[j / 2]
            const uint4& xa = x0[j >> 1];
            mma_bf16_16816(d[i][0], lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1],
                           (j & 1) ? xa.z : xa.x, (j & 1) ? xa.w : xa.y);
            if constexpr (kTwo) {
              const uint4& xb = x1[j >> 1];
              mma_bf16_16816(d[i][1], lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1],
                             (j & 1) ? xb.z : xb.x, (j & 1) ? xb.w : xb.y);
            }
          }
        }
      }
    }

    // D fragment of tile i, column tile c: d[0], d[1] = (row 16 i + g,
    // tokens 8 c + 2t, + 1), d[2], d[3] = row 16 i + g + 8.
#pragma unroll
    for (int i = 0; i < kTiles; ++i)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        red[warp][16 * i + g][8 * c + 2 * t] = d[i][c][0];
        red[warp][16 * i + g][8 * c + 2 * t + 1] = d[i][c][1];
        red[warp][16 * i + g + 8][8 * c + 2 * t] = d[i][c][2];
        red[warp][16 * i + g + 8][8 * c + 2 * t + 1] = d[i][c][3];
      }
    __syncthreads();
    {
      const int r = threadIdx.x & (kGroupRows - 1), m = threadIdx.x / kGroupRows;   // 32 x 16 outputs
      const int64_t n = row0 + r;
      if (m < M && n < r_end) {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < kWarps; ++q) acc += red[q][r][m];
        epi_store(out, static_cast<int64_t>(m) * N + n, ep.out_kind, epi_apply(ep, alpha * acc, n));
      }
    }
    __syncthreads();   // red is reused by the next row group
  }
}

template <int F>
cudaError_t launch_fewrow(const Ctx& c, void* out, const Epi& ep, const void* a,
                          const uint8_t* w, const uint8_t* bs, int64_t M, int64_t N, int64_t K,
                          float alpha) {
  // One CTA per SM with an even share of the rows (at least 8 each).
  int64_t grid = std::min<int64_t>(c.num_sms, (N + 7) / 8);
  if (grid < 1) grid = 1;
  const dim3 g(static_cast<unsigned>(grid)), b(kThreads);
  const auto* ab = static_cast<const uint16_t*>(a);
  const int m = static_cast<int>(M);
  if (M > 8)
    return launch_kernel(c, true, k_fewrow<F, true>, g, b, 0, out, ep, ab, w, bs, m, N, K, alpha);
  return launch_kernel(c, true, k_fewrow<F, false>, g, b, 0, out, ep, ab, w, bs, m, N, K, alpha);
}

}  // namespace

bool fewrow_ok(int format, int64_t M, int64_t K, const void* a, const uint8_t* w,
               const uint8_t* bs) {
  const int64_t step = format == kFewFp8 ? 64 : 128;
  if (M < 1 || M > kMaxM || K <= 0 || K % step != 0) return false;
  if (reinterpret_cast<uintptr_t>(a) % 16 != 0 || reinterpret_cast<uintptr_t>(w) % 16 != 0)
    return false;
  return format == kFewFp8 || reinterpret_cast<uintptr_t>(bs) % 2 == 0;
}

cudaError_t launch_fp8_gemm_fewrow(const Ctx& c, void* out, const Epi& ep, const void* a,
                                   const uint8_t* w, int64_t M, int64_t N, int64_t K,
                                   float alpha) {
  return launch_fewrow<kFewFp8>(c, out, ep, a, w, nullptr, M, N, K, alpha);
}

cudaError_t launch_nvfp4_gemm_fewrow(const Ctx& c, void* out, const Epi& ep, const void* a,
                                     const uint8_t* q, const uint8_t* bs, int64_t M, int64_t N,
                                     int64_t K, float alpha) {
  return launch_fewrow<kFewNvfp4>(c, out, ep, a, q, bs, M, N, K, alpha);
}

}  // namespace gq
