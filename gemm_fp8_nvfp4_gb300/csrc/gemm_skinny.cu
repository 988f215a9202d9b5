// gemm_skinny.cu -- the W8A16 / W4A16 GEMM for few activation rows (M <= 128)
// on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
//   C[m, n] = alpha * sum_k A[m, k] * w_hat[n, k]      (A bf16, fp32 accumulate)
//
// The contraction of gemm.cu (sources: the "fp4_matmul" kernel page -- packed
// weight tiles stay packed in memory and are dequantized to bf16 once per K
// strip in shared memory, where a dense bf16 MMA reads them; the "fp8_gemv"
// page -- the per-tensor scale is folded after the sum), organised for the
// decode-sized batches of the NVFP4 workload on the "fp4_matmul" page (M = 16
// and 128), where the weight is nearly all of the traffic and there are too
// few (M, N) tiles to fill the GPU:
//
// * One tile is all M rows (the MMA's M = 128; activation rows past M are
//   never loaded and only feed accumulator rows that are never stored) by TN
//   weight rows (the MMA's N), TN = 256 or 128.  A kind::f16 MMA with K = 16
//   takes the same time on the tensor core for every N up to 256 and for M =
//   64 or 128, so the weight sits on the N side, and TN = 256 halves the MMA
//   count; TN = 128 is used when 256-row tiles would leave SMs idle (with
//   half the dequant work per step, two groups of dequant warps then work on
//   alternate K steps).
// * K is split over a thread-block cluster of S <= 8 CTAs (any size whose
//   clusters are all resident at once) so that ceil(N / TN) * S CTAs fill the
//   GPU.  The fp32 partial tiles meet in distributed shared memory; rank r
//   sums its slice of ceil(TN / S) columns (rounded up to 4) of the tile over
//   the ranks in rank order (deterministic), scales, converts and stores them.
// * Three rings, each released by its own consumer: the raw weight ring,
//   freed as soon as its K steps are dequantized; the dequantized-weight
//   ring, freed by the MMA; and the activation ring with its own TMA warp,
//   freed by the MMA -- no TMA round trip sits inside the MMA's per-step loop.
// * A raw weight stage is 128 bytes of each of the TN rows (128-byte
//   swizzle): 4 K steps of NVFP4, 2 of FP8.  The TMA unit spends about the
//   same time on each row of a box whether the row is 32 or 128 bytes wide,
//   so narrow per-step boxes would cap the weight stream far below what the
//   MMA consumes.  NVFP4 block scales come by TMA too, 16 bytes per row per
//   raw stage (K a multiple of 256; other K go to the general kernel).
// * The weight is also prefetched into L2 kL2Ahead K steps ahead through a
//   second tensor map whose box is 256 bytes of each of the TN rows.
//
// Roles (24 warps):
//   warp 0        weight TMA producer (NVFP4: block scales by 4-byte cp.async)
//   warp 1        MMA issuer (one thread), TMEM owner
//   warp 2        activation TMA producer
//   warps 4..19   dequant: thread (row, half) decodes 32 K of one weight row;
//                 one group of 16 warps per K step (TN = 256) or two groups
//                 of 8 on alternate K steps (TN = 128)
//   warps 20..23  epilogue: TMEM -> fp32 partial tile in shared memory
//   all warps     cluster reduction, scale, convert, store
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gq {
namespace {

constexpr int UMMA_M = 128;       // activation rows per MMA (rows >= M are padding)
constexpr int BK = 64;            // K per stage (one 128-byte swizzle row of bf16)
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kMaxRows = UMMA_M;  // activation rows served by this kernel
constexpr int kL2Ahead = 32;      // weight K steps prefetched into L2 ahead of the ring
constexpr int kMinRawPerSplit = 2;  // each cluster rank gets at least this many raw stages
constexpr int kMaxSplit = 8;      // portable cluster size
constexpr int kThreads = 768;
constexpr int kWarpW = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpAct = 2;
constexpr int kDeqWarp0 = 4;
constexpr int kDeqWarps = 16;     // 512 threads: (row, half) pairs of one or two K steps
constexpr int kEpiWarp0 = 20;     // 4 warps: TMEM lane groups 0..3
constexpr uint32_t kActBytes = UMMA_M * BK * 2;   // 16 KB (rows >= M never written)
constexpr uint32_t kRawRow = 128;                 // weight bytes per row per raw stage

static_assert(kEpiWarp0 % 4 == 0, "epilogue warp w reads TMEM lanes 32 * (w % 4)");
static_assert(kDeqWarp0 + kDeqWarps <= kEpiWarp0 && kEpiWarp0 + 4 == kThreads / 32, "warp roles");

// Per tile size: ring depths and dequant warp groups.
template <int TN> struct TileCfg;
template <> struct TileCfg<256> {
  static constexpr int kDq = 2, kAct = 3, kRaw = 3, kGroups = 1;
};
template <> struct TileCfg<128> {
  static constexpr int kDq = 4, kAct = 4, kRaw = 4, kGroups = 2;
};

enum class Fmt { kFp8, kNvfp4 };

template <Fmt F> struct Raw;
template <> struct Raw<Fmt::kFp8> {
  static constexpr int kKbPer = 2;                          // K steps per raw stage
  static constexpr uint32_t kBpk = BK;                      // weight bytes per row per K step
  static constexpr uint32_t kSBytes = 0;
};
template <> struct Raw<Fmt::kNvfp4> {
  static constexpr int kKbPer = 4;
  static constexpr uint32_t kBpk = BK / 2;
  static constexpr uint32_t kSRow = 16;                     // scale bytes per row per raw stage
};

// Shared-memory layout (offsets from a 1 KB aligned base).  The dequant,
// activation and raw rings are adjacent: the fp32 partial tile reuses them.
template <Fmt F, int TN> struct Smem {
  using C = TileCfg<TN>;
  static constexpr uint32_t kDeqBytes = TN * BK * 2;          // bf16 weight tile per K step
  static constexpr uint32_t kRawBytes = TN * kRawRow;         // raw weight per raw stage
  static constexpr uint32_t kSBytes = F == Fmt::kNvfp4 ? TN * 16 : 0;   // block scales
  static constexpr uint32_t kPartStride = TN * 4 + 16;        // fp32 partial row + pad (banks)
  static constexpr uint32_t kDeqOff = 0;
  static constexpr uint32_t kActOff = kDeqOff + C::kDq * kDeqBytes;
  static constexpr uint32_t kRawOff = kActOff + C::kAct * kActBytes;
  static constexpr uint32_t kSclOff = kRawOff + C::kRaw * kRawBytes;
  static constexpr uint32_t kBarOff = (kSclOff + C::kRaw * kSBytes + 7) & ~7u;
  static constexpr uint32_t kNumBars = 2 * C::kRaw + 2 * C::kAct + 2 * C::kDq + 2;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;   // TMEM address, abort flag
  static constexpr uint32_t kAlloc = kMiscOff + 16 + 1024;        // + slack for 1 KB alignment
  static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
  static_assert(kMaxRows * kPartStride <= kSclOff, "the partial tile overlays the rings");
  static_assert(kDeqWarps / C::kGroups == 2 * TN / 32, "one (row, half) pair per dequant thread");
};

struct SkProblem {
  void* out;
  uint32_t* status;
  float alpha;
  int M, N, K;
  int m_pad;           // activation rows loaded per stage: M rounded up to 8
  int nkb;             // K steps of BK
  int ksplit;          // cluster size S (<= kMaxSplit)
  Epi ep;              // output type and fused epilogue
  int wp_box;          // inner box (bytes) of the weight prefetch map
  int overlap_weights; // the weight producer reads before the previous kernel completes
};

template <Fmt F, int TN>
__global__ void __launch_bounds__(kThreads, 1)
k_wq_gemm_skinny(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                 const __grid_constant__ CUtensorMap tmap_wp, const __grid_constant__ CUtensorMap tmap_s,
                 SkProblem p) {
  using R = Raw<F>;
  using L = Smem<F, TN>;
  using C = TileCfg<TN>;
  // Programmatic dependent launch: the next kernel in the stream may start
  // its launch now; this one sets up (barriers, TMEM, descriptors) while the
  // previous kernel finishes, and waits for it before any global access --
  // except, with GQ_LAUNCH_OVERLAP_WEIGHT_READS, the weight producer, whose
  // reads of the (unchanging) weights then overlap the previous kernel.
  pdl_launch_dependents();
  constexpr int kRawStages = C::kRaw, kActStages = C::kAct, kDqStages = C::kDq, kGroups = C::kGroups;
  constexpr uint32_t kRawBytes = L::kRawBytes, kDeqBytes = L::kDeqBytes, kPartStride = L::kPartStride;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full_raw = bars;
  uint64_t* empty_raw = full_raw + kRawStages;
  uint64_t* full_act = empty_raw + kRawStages;
  uint64_t* empty_act = full_act + kActStages;
  uint64_t* full_deq = empty_act + kActStages;
  uint64_t* empty_deq = full_deq + kDqStages;
  uint64_t* acc_full = empty_deq + kDqStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = tc::smem_u32(smem);

  const int S = p.ksplit;
  const int rank = static_cast<int>(blockIdx.x) % S;   // cluster dims (S, 1, 1)
  const int n0 = (static_cast<int>(blockIdx.x) / S) * TN;
  // Even split of the raw stages (kKbPer K steps each): every rank gets floor
  // or ceil of nrs / S of them, so its K steps start on a raw-stage boundary.
  const int nrs = (p.nkb + R::kKbPer - 1) / R::kKbPer;
  const int rs0 = static_cast<int>((static_cast<int64_t>(rank) * nrs) / S);
  const int rs1 = static_cast<int>((static_cast<int64_t>(rank + 1) * nrs) / S);
  const int nr = rs1 - rs0;
  const int kb0 = rs0 * R::kKbPer;
  const int kb1 = min(p.nkb, rs1 * R::kKbPer);
  const int nk = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      tc::mbar_init(&full_raw[s], 1);
      tc::mbar_init(&empty_raw[s], kDeqWarps);
    }
    for (int a = 0; a < kActStages; ++a) {
      tc::mbar_init(&full_act[a], 1);
      tc::mbar_init(&empty_act[a], 1);
    }
    for (int d = 0; d < kDqStages; ++d) {
      tc::mbar_init(&full_deq[d], kDeqWarps / kGroups);
      tc::mbar_init(&empty_deq[d], 1);
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(tmem_slot, TN);
    tc::tmem_relinquish();
  }
  if (warp == kWarpW && lane == 0) {
    tc::tma_prefetch_desc(&tmap_a);
    tc::tma_prefetch_desc(&tmap_w);
    tc::tma_prefetch_desc(&tmap_wp);
    if constexpr (F == Fmt::kNvfp4) tc::tma_prefetch_desc(&tmap_s);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool early_weights = p.overlap_weights && warp == kWarpW;
  if (!early_weights) pdl_wait();
  const uint32_t part = smem_base;   // fp32 partial tile [m][TN n], over the rings

  if (warp == kWarpW) {
    // ---------------------------------------------------- weight producer --
    if (lane == 0) {
      // The L2 prefetch cursor px walks this rank's byte range of the rows,
      // [kb0 * kBpk, kb1 * kBpk), in wp_box steps (x a multiple of 16 bytes).
      int px = kb0 * static_cast<int>(R::kBpk);
      auto prefetch_w_upto = [&](int kb_end) {
        const int lim = min(kb_end, kb1) * static_cast<int>(R::kBpk);
        for (; px < lim; px += p.wp_box) tc::tma_prefetch_l2_2d(&tmap_wp, px, n0);
      };
      // The first wide box goes out before the ring's own loads (which ride
      // on it); the rest of the prefetch follows once the ring is filled.
      prefetch_w_upto(kb0 + 1);
      int issued = 0;
      for (int j = 0; j < nr; ++j) {
        const int s = j % kRawStages;
        if (!tc::mbar_wait(&empty_raw[s], ((j / kRawStages) & 1) ^ 1, abort_flag, p.status,
                           kStatusTimeoutProducer))
          break;
        const int rs = rs0 + j;
        tc::mbar_arrive_expect_tx(&full_raw[s], kRawBytes + L::kSBytes);
        tc::tma_load_2d(smem + L::kRawOff + s * kRawBytes, &tmap_w, &full_raw[s],
                        rs * static_cast<int>(kRawRow), n0);
        if constexpr (F == Fmt::kNvfp4)
          tc::tma_load_2d(smem + L::kSclOff + s * L::kSBytes, &tmap_s, &full_raw[s],
                          rs * static_cast<int>(R::kSRow), n0);
        if (j + 1 >= min(nr, kRawStages)) prefetch_w_upto(min(kb1, (rs + 1) * R::kKbPer) + kL2Ahead);
        issued = j + 1;
      }
      // Drain: no copy may still be landing when the CTA exits (bounded;
      // normally complete already).
      for (int j = std::max(0, issued - kRawStages); j < issued; ++j)
        tc::mbar_wait_quiet(&full_raw[j % kRawStages], (j / kRawStages) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kWarpAct) {
    // ------------------------------------------------ activation producer --
    if (lane == 0) {
      // Only the first m_pad rows of a stage are loaded; the TMA box has
      // m_pad rows, so exactly that many bytes arrive.
      const uint32_t act_bytes = static_cast<uint32_t>(p.m_pad) * BK * 2;
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int a = i % kActStages;
        const uint32_t ph = (i / kActStages) & 1;
        if (!tc::mbar_wait(&empty_act[a], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
        tc::mbar_arrive_expect_tx(&full_act[a], act_bytes);
        tc::tma_load_2d(smem + L::kActOff + a * kActBytes, &tmap_a, &full_act[a], (kb0 + i) * BK, 0);
        issued = i + 1;
      }
      for (int i = std::max(0, issued - kActStages); i < issued; ++i)
        tc::mbar_wait_quiet(&full_act[i % kActStages], (i / kActStages) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer --
    constexpr uint32_t kIdesc = tc::idesc_bf16_f32(UMMA_M, TN);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int d = i % kDqStages;
      const int a = i % kActStages;
      if (!tc::mbar_wait(&full_act[a], (i / kActStages) & 1, abort_flag, p.status, kStatusTimeoutMma) ||
          !tc::mbar_wait(&full_deq[d], (i / kDqStages) & 1, abort_flag, p.status, kStatusTimeoutMma)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      if (lane == 0) {
        const uint32_t x_addr = smem_base + L::kActOff + a * kActBytes;
        const uint32_t w_addr = smem_base + L::kDeqOff + d * kDeqBytes;
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t ad = tc::sw128_kmajor_desc(x_addr + kk * UMMA_K * 2);
          const uint64_t bd = tc::sw128_kmajor_desc(w_addr + kk * UMMA_K * 2);
          tc::mma_bf16(tmem_base, ad, bd, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&empty_deq[d]);
        tc::mma_commit(&empty_act[a]);
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
    // Group grp takes the K steps i = grp (mod kGroups); within a group,
    // thread (row, half) decodes K elements [32 * half, 32 * half + 32) of
    // weight row `row` of the step.
    constexpr int kWarpsPerGroup = kDeqWarps / kGroups;
    const int w = warp - kDeqWarp0;
    const int grp = w / kWarpsPerGroup;
    const int wg = w % kWarpsPerGroup;
    const int row = (wg % (TN / 32)) * 32 + lane;
    const int half = wg / (TN / 32);
    for (int i = grp; i < nk; i += kGroups) {
      const int j = i / R::kKbPer;           // raw stage of this rank
      const int sub = i % R::kKbPer;         // K step within it
      const int s = j % kRawStages;
      const int d = i % kDqStages;
      const bool first_in_stage = i < kGroups || (i - kGroups) / R::kKbPer != j;
      const bool last_in_stage = i + kGroups >= nk || (i + kGroups) / R::kKbPer != j;
      if ((first_in_stage && !tc::mbar_wait(&full_raw[s], (j / kRawStages) & 1, abort_flag, p.status,
                                            kStatusTimeoutDequant)) ||
          !tc::mbar_wait(&empty_deq[d], ((i / kDqStages) & 1) ^ 1, abort_flag, p.status,
                         kStatusTimeoutDequant))
        break;
      // Raw row: 128 bytes, 128-byte swizzle -- 16-byte chunk c at c ^ (row & 7).
      const uint32_t w_row = smem_base + L::kRawOff + s * kRawBytes + row * kRawRow;
      const uint32_t b_addr = smem_base + L::kDeqOff + d * kDeqBytes;
      if constexpr (F == Fmt::kFp8) {
        // Step sub = bytes [64 * sub, 64 * sub + 64) of the row: chunks 4 sub .. 4 sub + 3.
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 4 * sub + 2 * half + c2;
          const uint4 v = tc::lds128(w_row + ((c ^ (row & 7)) << 4));
          uint4 lo, hi;
          fp8x16_to_bf16(v, lo, hi);
          tc::sts128(b_addr + sw128_off(row, 4 * half + 2 * c2), lo);
          tc::sts128(b_addr + sw128_off(row, 4 * half + 2 * c2 + 1), hi);
        }
      } else {
        // Step sub = bytes [32 * sub, 32 * sub + 32): chunk 2 sub + half holds
        // this thread's 32 codes; block scales 2 * half, 2 * half + 1 of the
        // step's four are bytes 4 sub + 2 half, + 1 of the row's 16.
        const uint32_t sc =
            tc::lds32(smem_base + L::kSclOff + s * L::kSBytes + row * R::kSRow + sub * 4);
        const int c = 2 * sub + half;
        const uint4 v = tc::lds128(w_row + ((c ^ (row & 7)) << 4));
        const uint16_t s0 = e4m3_to_f16(sc >> (16 * half));
        const uint16_t s1 = e4m3_to_f16(sc >> (16 * half + 8));
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
        if (last_in_stage) tc::mbar_arrive(&empty_raw[s]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue --
    // TMEM lane m (activation row), column n -> partial[m][n] (fp32).  The
    // dequant and activation rings are idle: every MMA has completed when
    // acc_full fires.  Warps whose rows are all >= M skip the copy.
    const int g = warp & 3;
    const int m = g * 32 + lane;
    if (g * 32 < p.M && tc::mbar_wait(acc_full, 0, abort_flag, p.status, kStatusTimeoutEpilogue)) {
      tc::tc_fence_after();
      const uint32_t prow = part + m * kPartStride;
#pragma unroll 1
      for (int c0 = 0; c0 < TN; c0 += 32) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(g * 32) << 16) + c0, r);
        tc::tmem_wait_ld();
        if (m < p.M) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            tc::sts128(prow + (c0 + 4 * i) * 4, make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]));
        }
      }
    }
  }

  if (early_weights) pdl_wait();   // before this warp's part of the output stores
  tc::tc_fence_before();
  __syncthreads();
  if (S > 1) tc::cluster_sync();
  {
    // Rank r: columns [r * cols, min(TN, (r + 1) * cols)) of the tile, all
    // M rows, four columns per task.
    const int cols = ((TN + S - 1) / S + 3) / 4 * 4;
    const int c_end = min(TN, (rank + 1) * cols);
    const int per_row = cols / 4;
    const int tasks = p.M * per_row;
    const bool vec = (p.N & 3) == 0;
    for (int task = threadIdx.x; task < tasks; task += kThreads) {
      const int m = task / per_row;
      const int nl = rank * cols + 4 * (task % per_row);
      const int n = n0 + nl;
      if (nl >= c_end || n >= p.N) continue;
      const uint32_t addr = part + m * kPartStride + nl * 4;
      float4 acc;
      if (S == 1) {
        acc = tc::lds_f4(addr);
      } else {
        // every rank's partial requested before the first add (the loads are
        // in flight together), then summed in rank order
        float4 v[kMaxSplit];
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
          if (q < S) v[q] = tc::ld_cluster_f4(tc::map_to_rank(addr, q));
        acc = v[0];
#pragma unroll
        for (int q = 1; q < kMaxSplit; ++q) {
          if (q < S) {
            acc.x += v[q].x; acc.y += v[q].y; acc.z += v[q].z; acc.w += v[q].w;
          }
        }
      }
      const int lim = min(4, p.N - n);
      float o[4] = {p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = epi_apply(p.ep, o[i], n + (i < lim ? i : 0));
      const int64_t base = static_cast<int64_t>(m) * p.N + n;
      if (vec && lim == 4) {
        epi_store4(p.out, base, p.ep.out_kind, o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < lim) epi_store(p.out, base + i, p.ep.out_kind, o[i]);
      }
    }
  }
  // No CTA leaves while a peer still reads its partial.  The peers' reads
  // have returned (their values were used) before they arrive, so the
  // barrier needs no memory ordering -- and a release here would wait for
  // this thread's global stores.
  if (S > 1) tc::cluster_sync_relaxed();
  if (warp == kWarpMma) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, TN);
  }
}

// --------------------------------------------------------------- host --

// The shared-memory opt-in, set once per device and kernel.
template <Fmt F, int TN>
cudaError_t configure(int device) {
  static std::atomic<uint64_t> done{0};
  const uint64_t bit = 1ull << (device & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_wq_gemm_skinny<F, TN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<F, TN>::kAlloc);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// How many clusters of S CTAs can be resident at once; cached, the answer
// depends only on the device, the kernel and the cluster size.
template <Fmt F, int TN>
int max_active_clusters(int device, int S) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;
  const auto key = std::make_pair(device, S);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (configure<F, TN>(device) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Smem<F, TN>::kAlloc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k_wq_gemm_skinny<F, TN>, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

// K split for TN-row tiles: the largest S <= kMaxSplit such that the tiles *
// S CTAs fit on the GPU in one wave (all clusters resident at once) and every
// rank keeps at least kMinRawPerSplit raw stages.
template <Fmt F, int TN>
int plan_split(const Ctx& c, int tiles, int nkb) {
  const int nrs = (nkb + Raw<F>::kKbPer - 1) / Raw<F>::kKbPer;
  for (int S = kMaxSplit; S > 1; --S) {
    if (tiles * S > c.num_sms || nrs < S * kMinRawPerSplit) continue;
    if (max_active_clusters<F, TN>(c.device, S) >= tiles) return S;
  }
  return 1;
}

// Tensor maps for TN-row tiles.  The weight rows are row_bytes long: raw
// stages of 128 bytes (128-byte swizzle) and L2 prefetch boxes of up to 256
// bytes; NVFP4 block scales in boxes of 16 bytes (K / 16 bytes per row).
template <Fmt F, int TN>
bool encode_maps(SkProblem& p, const void* a, const uint8_t* w, const uint8_t* bs, int64_t row_bytes,
                 CUtensorMap* ta, CUtensorMap* tw, CUtensorMap* twp, CUtensorMap* ts) {
  p.wp_box = static_cast<int>(std::min<int64_t>(256, row_bytes));   // a multiple of 16
  if (!encode_2d(ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, p.K, p.M, static_cast<int64_t>(p.K) * 2, BK,
                 p.m_pad, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, p.N, row_bytes, kRawRow, TN,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(twp, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, p.N, row_bytes, p.wp_box, TN,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  memset(ts, 0, sizeof(*ts));
  if constexpr (F == Fmt::kNvfp4) {
    const int64_t ks = p.K / 16;
    if (!encode_2d(ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, bs, ks, p.N, ks, Raw<F>::kSRow, TN,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
  }
  return true;
}

template <Fmt F, int TN>
cudaError_t launch_tn(const Ctx& c, SkProblem p, int S, const void* a, const uint8_t* w,
                      const uint8_t* bs, int64_t row_bytes) {
  if (cudaError_t e = configure<F, TN>(c.device)) return e;
  CUtensorMap ta, tw, twp, ts;
  if (!encode_maps<F, TN>(p, a, w, bs, row_bytes, &ta, &tw, &twp, &ts)) return cudaErrorInvalidValue;
  p.ksplit = S;
  const int tiles = (p.N + TN - 1) / TN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<F, TN>::kAlloc;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = S > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_wq_gemm_skinny<F, TN>, ta, tw, twp, ts, p);
}

// 256-row tiles halve the MMA count; 128-row tiles are used when they keep
// more SMs busy (few N tiles).
template <Fmt F>
cudaError_t launch(const Ctx& c, SkProblem p, const void* a, const uint8_t* w, const uint8_t* bs,
                   int64_t row_bytes) {
  const int tiles256 = (p.N + 255) / 256;
  const int tiles128 = (p.N + 127) / 128;
  const int s256 = plan_split<F, 256>(c, tiles256, p.nkb);
  const int s128 = plan_split<F, 128>(c, tiles128, p.nkb);
  if (tiles256 * s256 >= tiles128 * s128) return launch_tn<F, 256>(c, p, s256, a, w, bs, row_bytes);
  return launch_tn<F, 128>(c, p, s128, a, w, bs, row_bytes);
}

SkProblem make_problem(const Ctx& c, void* out, const Epi& ep, int64_t M, int64_t N, int64_t K,
                       float alpha) {
  SkProblem p{};
  p.out = out;
  p.status = c.status;
  p.alpha = alpha;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_pad = static_cast<int>((M + 7) / 8 * 8);
  p.nkb = static_cast<int>((K + BK - 1) / BK);
  p.ksplit = 1;
  p.ep = ep;
  p.overlap_weights = c.overlap_weights ? 1 : 0;
  return p;
}

}  // namespace

int skinny_max_rows() { return kMaxRows; }

bool nvfp4_skinny_ok(const uint8_t* bs, int64_t K) {
  // Block scales by TMA: 16-byte rows (K / 16 a multiple of 16) and base.
  return K % 256 == 0 && (reinterpret_cast<uintptr_t>(bs) & 15) == 0;
}

cudaError_t launch_fp8_gemm_skinny(const Ctx& c, void* out, const Epi& ep, const void* a,
                                   const uint8_t* w, int64_t M, int64_t N, int64_t K, float alpha) {
  return launch<Fmt::kFp8>(c, make_problem(c, out, ep, M, N, K, alpha), a, w, nullptr, K);
}

cudaError_t launch_nvfp4_gemm_skinny(const Ctx& c, void* out, const Epi& ep, const void* a,
                                     const uint8_t* q, const uint8_t* bs, int64_t M, int64_t N,
                                     int64_t K, float alpha) {
  if (!nvfp4_skinny_ok(bs, K)) return cudaErrorInvalidValue;
  return launch<Fmt::kNvfp4>(c, make_problem(c, out, ep, M, N, K, alpha), a, q, bs, K / 2);
}

}  // namespace gq
