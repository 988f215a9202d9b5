// gemm_skinny.cu -- the W8A16 / W4A16 GEMM for few activation rows (M <= 128)
// on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
//   C[m, n] = alpha * sum_k A[m, k] * w_hat[n, k]      (A bf16, fp32 accumulate)
//
// The contraction of gemm.cu (sources: the "fp4_matmul" kernel page -- packed
// weight tiles stay packed in memory and are dequantized to bf16 once per K
// strip in shared memory, where a dense bf16 MMA reads them; the "fp8_gemv"
// page -- the per-tensor scale is folded after the sum), organised for the
// decode-sized batches of the NVFP4 workload on the "fp4_matmul" page
// (M = 16 and 128), where the weight is nearly all of the traffic and a
// 256-row activation tile would leave the tensor core computing padding:
//
// * Operand roles swapped.  The dequantized weight tile (128 weight rows x 64
//   K) is the MMA's A operand (M = 128); the activation rows are the B operand
//   (N = M rounded up to 16).  TMEM holds the transposed tile: lane = output
//   column n, TMEM column = output row m.
// * K split over a thread-block cluster of S CTAs, S a power of two, so that
//   ceil(N / 128) * S CTAs fill the GPU.  The fp32 partial tiles meet in
//   distributed shared memory; rank r sums columns [r * 128 / S, (r + 1) *
//   128 / S) of the tile over the ranks in rank order (deterministic), scales,
//   converts and stores them.
// * The raw weight ring is deep (16 stages NVFP4, 8 FP8) and a stage is
//   released as soon as it is dequantized, independently of the MMA; the
//   activation tiles have their own TMA warp and ring, tied to the dequant
//   ring.  Weight tiles are prefetched into L2 kL2Ahead K steps ahead.
//
// Roles (16 warps):
//   warp 0       weight TMA producer (NVFP4: block scales by 4-byte cp.async)
//   warp 1       MMA issuer (one thread), TMEM owner
//   warp 2       activation TMA producer
//   warps 4..11  dequant: thread (row, half) decodes 32 K of one weight row
//   warps 12..15 epilogue: TMEM -> fp32 partial tile in shared memory
//   all warps    cluster reduction, scale, convert, store
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gq {
namespace {

constexpr int kTileN = 128;       // weight rows per tile (the MMA's M)
constexpr int BK = 64;            // K per stage (one 128-byte swizzle row of bf16)
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kMaxRows = 128;     // activation rows served by this kernel
constexpr int kDqStages = 4;      // dequantized-weight / activation stages
constexpr int kL2Ahead = 32;      // weight K steps prefetched into L2 ahead of the ring
constexpr int kMinKbPerSplit = 4; // each cluster rank gets at least this many K steps
constexpr int kMaxSplit = 8;      // portable cluster size
constexpr int kThreads = 512;
constexpr int kWarpW = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpAct = 2;
constexpr int kDeqWarp0 = 4;
constexpr int kDeqWarps = 8;      // 256 threads: (row, half) pairs of the 128-row tile
constexpr int kEpiWarp0 = 12;     // 4 warps: TMEM lane groups 0..3

constexpr uint32_t kDeqBytes = kTileN * BK * 2;   // 16 KB
constexpr uint32_t kActRowBytes = BK * 2;         // 128 B per activation row per stage
constexpr uint32_t kPartRow = kTileN * 4;         // 512 B: one output row of the fp32 partial

static_assert(kMaxRows * kPartRow <= kDqStages * kDeqBytes,
              "the partial tile overlays the dequant ring");

enum class Fmt { kFp8, kNvfp4 };

template <Fmt F> struct Raw;
template <> struct Raw<Fmt::kFp8> {
  static constexpr int kStages = 8;
  static constexpr uint32_t kWBytes = kTileN * BK;          // 8 KB, 64-byte swizzle
  static constexpr uint32_t kSBytes = 0;
};
template <> struct Raw<Fmt::kNvfp4> {
  static constexpr int kStages = 16;
  static constexpr uint32_t kWBytes = kTileN * BK / 2;      // 4 KB, 32-byte swizzle
  static constexpr uint32_t kSBytes = kTileN * BK / 16;     // 512 B: 4 scale bytes per row
};

// Shared-memory layout for m_pad activation rows (offsets from a 1 KB aligned base).
template <Fmt F> struct Layout {
  static constexpr uint32_t kNumBars = 2 * Raw<F>::kStages + 3 * kDqStages + 2;
  uint32_t act, raw, scl, bar, misc, total;
  __host__ __device__ explicit Layout(int m_pad) {
    act = kDqStages * kDeqBytes;
    raw = act + kDqStages * static_cast<uint32_t>(m_pad) * kActRowBytes;
    scl = raw + Raw<F>::kStages * Raw<F>::kWBytes;
    bar = (scl + Raw<F>::kStages * Raw<F>::kSBytes + 7) & ~7u;
    misc = bar + kNumBars * 8;   // TMEM address, abort flag
    total = misc + 16;
  }
};

struct SkProblem {
  void* out;
  uint32_t* status;
  float alpha;
  int M, N, K;
  int m_pad;           // M rounded up to 16: the MMA's N
  int nkb;             // K steps of BK
  int ksplit;          // cluster size S (power of two, <= kMaxSplit)
  int bf16_out;
  int scale_prefetch;  // NVFP4: the block-scale tensor map is valid (L2 prefetch)
};

template <Fmt F>
__global__ void __launch_bounds__(kThreads, 1)
k_wq_gemm_skinny(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_s, const uint8_t* __restrict__ scales_g,
                 SkProblem p) {
  using R = Raw<F>;
  const Layout<F> L(p.m_pad);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* full_raw = bars;
  uint64_t* empty_raw = full_raw + R::kStages;
  uint64_t* full_act = empty_raw + R::kStages;
  uint64_t* full_deq = full_act + kDqStages;
  uint64_t* empty_dq = full_deq + kDqStages;   // MMA done with dequant + activation stage
  uint64_t* acc_full = empty_dq + kDqStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = tc::smem_u32(smem);

  const int S = p.ksplit;
  const int rank = static_cast<int>(blockIdx.x) % S;   // cluster dims (S, 1, 1)
  const int n0 = (static_cast<int>(blockIdx.x) / S) * kTileN;
  // Even split of the K steps: every rank gets floor or ceil of nkb / S (>= 1).
  const int kb0 = static_cast<int>((static_cast<int64_t>(rank) * p.nkb) / S);
  const int kb1 = static_cast<int>((static_cast<int64_t>(rank + 1) * p.nkb) / S);
  const int nk = kb1 - kb0;
  const uint32_t tmem_cols = p.m_pad <= 32 ? 32u : (p.m_pad <= 64 ? 64u : 128u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < R::kStages; ++s) {
      tc::mbar_init(&full_raw[s], F == Fmt::kNvfp4 ? 1 + 32 : 1);
      tc::mbar_init(&empty_raw[s], kDeqWarps);
    }
    for (int d = 0; d < kDqStages; ++d) {
      tc::mbar_init(&full_act[d], 1);
      tc::mbar_init(&full_deq[d], kDeqWarps);
      tc::mbar_init(&empty_dq[d], 1);
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(tmem_slot, tmem_cols);
    tc::tmem_relinquish();
  }
  if (warp == kWarpW && lane == 0) {
    tc::tma_prefetch_desc(&tmap_a);
    tc::tma_prefetch_desc(&tmap_w);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t part = smem_base;   // fp32 partial tile [m][128 n], over the dequant ring

  if (warp == kWarpW) {
    // ---------------------------------------------------- weight producer --
    auto prefetch_w = [&](int kb) {
      if constexpr (F == Fmt::kFp8) tc::tma_prefetch_l2_2d(&tmap_w, kb * BK, n0);
      else tc::tma_prefetch_l2_2d(&tmap_w, kb * (BK / 2), n0);
    };
    if (lane == 0) {
      for (int kb = kb0; kb < kb1 && kb < kb0 + kL2Ahead; ++kb) prefetch_w(kb);
      if constexpr (F == Fmt::kNvfp4) {
        // This rank's block scales: 4 bytes per row per K step, boxes of 64
        // bytes (x stays a multiple of 16 bytes).
        if (p.scale_prefetch)
          for (int x = (kb0 * 4) & ~63; x < kb1 * 4; x += 64) tc::tma_prefetch_l2_2d(&tmap_s, x, n0);
      }
    }
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int kb = kb0 + i;
      const int s = i % R::kStages;
      const uint32_t ph = (i / R::kStages) & 1;
      if (lane == 0 && kb + kL2Ahead < kb1) prefetch_w(kb + kL2Ahead);
      if (!tc::mbar_wait(&empty_raw[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
      uint8_t* w_dst = smem + L.raw + s * R::kWBytes;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(&full_raw[s], R::kWBytes);
        if constexpr (F == Fmt::kFp8) tc::tma_load_2d(w_dst, &tmap_w, &full_raw[s], kb * BK, n0);
        else tc::tma_load_2d(w_dst, &tmap_w, &full_raw[s], kb * (BK / 2), n0);
      }
      if constexpr (F == Fmt::kNvfp4) {
        uint8_t* s_dst = smem + L.scl + s * R::kSBytes;
        const int64_t ks = p.K / 16;
#pragma unroll
        for (int j = 0; j < kTileN / 32; ++j) {
          const int r = lane + 32 * j;
          const int n = n0 + r;
          const bool in = n < p.N;
          tc::cp_async_4(s_dst + r * 4, scales_g + ((in ? n : 0) * ks + kb * 4), in ? 4u : 0u);
        }
        tc::cp_async_mbar_arrive_noinc(&full_raw[s]);
      }
      issued = i + 1;
    }
    // Drain: no copy of this warp may still be landing when the CTA exits
    // (bounded; normally complete already).
    if (lane == 0) {
      for (int i = std::max(0, issued - R::kStages); i < issued; ++i)
        tc::mbar_wait_quiet(&full_raw[i % R::kStages], (i / R::kStages) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kWarpAct) {
    // ------------------------------------------------ activation producer --
    if (lane == 0) {
      const uint32_t act_bytes = static_cast<uint32_t>(p.m_pad) * kActRowBytes;
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int d = i % kDqStages;
        const uint32_t ph = (i / kDqStages) & 1;
        if (!tc::mbar_wait(&empty_dq[d], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
        tc::mbar_arrive_expect_tx(&full_act[d], act_bytes);
        tc::tma_load_2d(smem + L.act + d * act_bytes, &tmap_a, &full_act[d], (kb0 + i) * BK, 0);
        issued = i + 1;
      }
      for (int i = std::max(0, issued - kDqStages); i < issued; ++i)
        tc::mbar_wait_quiet(&full_act[i % kDqStages], (i / kDqStages) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer --
    const uint32_t idesc = tc::idesc_bf16_f32(kTileN, p.m_pad);
    const uint32_t act_bytes = static_cast<uint32_t>(p.m_pad) * kActRowBytes;
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int d = i % kDqStages;
      const uint32_t ph = (i / kDqStages) & 1;
      if (!tc::mbar_wait(&full_act[d], ph, abort_flag, p.status, kStatusTimeoutMma) ||
          !tc::mbar_wait(&full_deq[d], ph, abort_flag, p.status, kStatusTimeoutMma)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      if (lane == 0) {
        const uint32_t w_addr = smem_base + d * kDeqBytes;
        const uint32_t x_addr = smem_base + L.act + d * act_bytes;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t ad = tc::sw128_kmajor_desc(w_addr + kk * UMMA_K * 2);
          const uint64_t bd = tc::sw128_kmajor_desc(x_addr + kk * UMMA_K * 2);
          tc::mma_bf16(tmem_base, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&empty_dq[d]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (ok && nk > 0) tc::mma_commit(acc_full);
      // Every MMA of this thread completes before TMEM is freed.
      tc::mma_commit(drain);
      tc::mbar_wait_quiet(drain, 0, 100000000ull);
    }
    __syncwarp();
  } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // -------------------------------------------------------------- dequant --
    const int w = warp - kDeqWarp0;
    const int row = (w & 3) * 32 + lane;   // weight row in the tile
    const int half = w >> 2;               // K elements [32 * half, 32 * half + 32) of the stage
    for (int i = 0; i < nk; ++i) {
      const int s = i % R::kStages;
      const int d = i % kDqStages;
      if (!tc::mbar_wait(&full_raw[s], (i / R::kStages) & 1, abort_flag, p.status, kStatusTimeoutDequant) ||
          !tc::mbar_wait(&empty_dq[d], ((i / kDqStages) & 1) ^ 1, abort_flag, p.status,
                         kStatusTimeoutDequant))
        break;
      const uint32_t w_addr = smem_base + L.raw + s * R::kWBytes;
      const uint32_t b_addr = smem_base + d * kDeqBytes;
      if constexpr (F == Fmt::kFp8) {
        // Row of 64 codes, TMA 64-byte swizzle: chunk c sits at c ^ ((row >> 1) & 3).
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * half + c2;
          const uint4 v = tc::lds128(w_addr + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
          uint4 lo, hi;
          fp8x16_to_bf16(v, lo, hi);
          tc::sts128(b_addr + sw128_off(row, 2 * c), lo);
          tc::sts128(b_addr + sw128_off(row, 2 * c + 1), hi);
        }
      } else {
        // Row of 32 packed bytes, TMA 32-byte swizzle: chunk c at c ^ ((row >> 2) & 1);
        // block scales 2 * half and 2 * half + 1 of the stage's four.
        const uint32_t sc = tc::lds32(smem_base + L.scl + s * R::kSBytes + row * 4);
        const uint4 v = tc::lds128(w_addr + row * 32 + ((half ^ ((row >> 2) & 1)) << 4));
        const float s0 = e4m3_to_f32(sc >> (16 * half));
        const float s1 = e4m3_to_f32(sc >> (16 * half + 8));
        uint4 lo, hi;
        nvfp4x16_to_bf16(v.x, v.y, s0, lo, hi);
        tc::sts128(b_addr + sw128_off(row, 4 * half), lo);
        tc::sts128(b_addr + sw128_off(row, 4 * half + 1), hi);
        nvfp4x16_to_bf16(v.z, v.w, s1, lo, hi);
        tc::sts128(b_addr + sw128_off(row, 4 * half + 2), lo);
        tc::sts128(b_addr + sw128_off(row, 4 * half + 3), hi);
      }
      tc::fence_proxy_async_smem();   // generic stores -> visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&full_deq[d]);
        tc::mbar_arrive(&empty_raw[s]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue --
    // TMEM lane n, column m -> partial[m][n] (fp32).  The dequant ring is idle:
    // every MMA has completed when acc_full fires.
    const int g = warp & 3;
    const int nl = g * 32 + lane;
    if (tc::mbar_wait(acc_full, 0, abort_flag, p.status, kStatusTimeoutEpilogue)) {
      tc::tc_fence_after();
      for (int c0 = 0; c0 < p.m_pad; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(g * 32) << 16) + c0, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) tc::sts32(part + (c0 + j) * kPartRow + nl * 4, r[j]);
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (S > 1) tc::cluster_sync();
  {
    // Rank r: columns [r * cols, (r + 1) * cols) of the tile, all M rows,
    // four columns per task.
    const int cols = kTileN / S;
    const int per_row = cols / 4;
    const int tasks = p.M * per_row;
    const bool vec = (p.N & 3) == 0;
    for (int task = threadIdx.x; task < tasks; task += kThreads) {
      const int m = task / per_row;
      const int nl = rank * cols + 4 * (task % per_row);
      const int n = n0 + nl;
      if (n >= p.N) continue;
      const uint32_t addr = part + m * kPartRow + nl * 4;
      float4 acc;
      if (S == 1) {
        acc = tc::lds_f4(addr);
      } else {
        acc = tc::ld_cluster_f4(tc::map_to_rank(addr, 0));
#pragma unroll
        for (int q = 1; q < kMaxSplit; ++q) {
          if (q < S) {
            const float4 v = tc::ld_cluster_f4(tc::map_to_rank(addr, q));
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
        }
      }
      const float o[4] = {p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w};
      const int64_t base = static_cast<int64_t>(m) * p.N + n;
      if (vec && n + 4 <= p.N) {
        if (p.bf16_out) {
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + base) =
              make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(p.out) + base) = make_float4(o[0], o[1], o[2], o[3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (n + i < p.N) {
            if (p.bf16_out) static_cast<__nv_bfloat16*>(p.out)[base + i] = __float2bfloat16_rn(o[i]);
            else static_cast<float*>(p.out)[base + i] = o[i];
          }
        }
      }
    }
  }
  if (S > 1) tc::cluster_sync();   // no CTA leaves while a peer still reads its partial
  if (warp == kWarpMma) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, tmem_cols);
  }
}

// --------------------------------------------------------------- host --

template <Fmt F>
uint32_t smem_bytes(int m_pad) {
  return Layout<F>(m_pad).total + 1024;   // slack for the 1 KB alignment
}

// The shared-memory opt-in, set once per device for the largest layout.
template <Fmt F>
cudaError_t configure(int device) {
  static std::atomic<uint64_t> done{0};
  const uint64_t bit = 1ull << (device & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_wq_gemm_skinny<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes<F>(kMaxRows));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// How many clusters of S CTAs (with this shared-memory size) can be resident
// at once; cached, the answer depends only on the device and the launch shape.
template <Fmt F>
int max_active_clusters(int device, int S, uint32_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, uint32_t>, int> cache;
  const auto key = std::make_tuple(device, S, smem);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_wq_gemm_skinny<F>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

// K split: the largest power of two S <= kMaxSplit such that tiles * S CTAs
// fit on the GPU in one wave (as clusters) and every rank keeps at least
// kMinKbPerSplit K steps.
template <Fmt F>
int plan_split(const Ctx& c, int tiles, int nkb, uint32_t smem) {
  int S = 1;
  while (S < kMaxSplit && tiles * S * 2 <= c.num_sms && nkb >= S * 2 * kMinKbPerSplit) S *= 2;
  while (S > 1 && max_active_clusters<F>(c.device, S, smem) < tiles) S /= 2;
  return S;
}

template <Fmt F>
cudaError_t launch(const Ctx& c, const CUtensorMap& ta, const CUtensorMap& tw, const CUtensorMap& ts,
                   const uint8_t* scales, SkProblem p) {
  if (cudaError_t e = configure<F>(c.device)) return e;
  const uint32_t smem = smem_bytes<F>(p.m_pad);
  const int tiles = (p.N + kTileN - 1) / kTileN;
  p.ksplit = plan_split<F>(c, tiles, p.nkb, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * p.ksplit);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.ksplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.ksplit > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_wq_gemm_skinny<F>, ta, tw, ts, scales, p);
}

SkProblem make_problem(const Ctx& c, void* out, bool bf16_out, int64_t M, int64_t N, int64_t K,
                       float alpha) {
  SkProblem p{};
  p.out = out;
  p.status = c.status;
  p.alpha = alpha;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_pad = static_cast<int>((M + 15) / 16 * 16);
  p.nkb = static_cast<int>((K + BK - 1) / BK);
  p.ksplit = 1;
  p.bf16_out = bf16_out ? 1 : 0;
  return p;
}

bool encode_act(CUtensorMap* ta, const void* a, int64_t M, int64_t K, int m_pad) {
  return encode_2d(ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, M, K * 2, BK, m_pad,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

int skinny_max_rows() { return kMaxRows; }

cudaError_t launch_fp8_gemm_skinny(const Ctx& c, void* out, bool bf16_out, const void* a,
                                   const uint8_t* w, int64_t M, int64_t N, int64_t K, float alpha) {
  SkProblem p = make_problem(c, out, bf16_out, M, N, K, alpha);
  CUtensorMap ta, tw, ts;
  memset(&ts, 0, sizeof(ts));
  if (!encode_act(&ta, a, M, K, p.m_pad) ||
      !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, BK, kTileN, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  return launch<Fmt::kFp8>(c, ta, tw, ts, nullptr, p);
}

cudaError_t launch_nvfp4_gemm_skinny(const Ctx& c, void* out, bool bf16_out, const void* a,
                                     const uint8_t* q, const uint8_t* bs, int64_t M, int64_t N,
                                     int64_t K, float alpha) {
  SkProblem p = make_problem(c, out, bf16_out, M, N, K, alpha);
  CUtensorMap ta, tw, ts;
  memset(&ts, 0, sizeof(ts));
  if (!encode_act(&ta, a, M, K, p.m_pad) ||
      !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K / 2, N, K / 2, BK / 2, kTileN,
                 CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  // The block-scale map (L2 prefetch only) needs 16-byte rows and base.
  const int64_t ks = K / 16;
  if (ks % 16 == 0 && (reinterpret_cast<uintptr_t>(bs) & 15) == 0) {
    p.scale_prefetch = encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, bs, ks, N, ks,
                                 static_cast<uint32_t>(std::min<int64_t>(64, ks)), kTileN,
                                 CU_TENSOR_MAP_SWIZZLE_NONE)
                           ? 1
                           : 0;
  }
  return launch<Fmt::kNvfp4>(c, ta, tw, ts, bs, p);
}

}  // namespace gq
