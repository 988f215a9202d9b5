// gemm.cu -- W8A16 / W4A16 GEMMs, the grouped (MoE) GEMMs of both formats
// and the W8A8 int8 GEMM on the 5th-generation tensor cores (tcgen05) of
// sm_103a.
//
//   C[m, n] = alpha * sum_k A[m, k] * w_hat[n, k]      (A bf16, fp32 accumulate)
//
// Sources: the "fp4_matmul" kernel page (AppleM5Fp4MatMul: the packed weight
// stays packed in memory, each (BN, BK) weight sub-tile is dequantized to bf16
// once per K-strip into shared memory, cooperatively, and a dense bf16 MMA
// reads it from there; the weight is the B operand, stored [N, K] row-major);
// the "fp8_gemv" page (enqueue_apple_fp8_matmul: the raw W8A16 matmul with the
// per-tensor scale folded after it); the "Matmul2dFp8" page (run_grouped: one
// expert group per z, ragged rows from a_offsets, empty groups and out-of-range
// M tiles skipped, expert id -1 writes zeros, per-expert scale after the sum).
//
// GB300 design (one persistent CTA per SM, warp-specialized):
//   warp 0        TMA producer: A tile [256 x 64] bf16 (128-byte swizzle) and
//                 the raw weight tile [256 x 64 codes] (FP8) or
//                 [256 x 32 bytes] + block scales (NVFP4) into a ring of
//                 kRawStages shared-memory stages, completion via mbarriers.
//   warps 4..11   dequant: each thread owns one weight row of the tile, decodes
//                 it exactly to bf16 and writes it in the 128-byte-swizzled
//                 K-major layout the tensor core reads, into a ring of
//                 kDeqStages stages.  Replaces the pages' barrier-fenced
//                 cooperative decode; here it overlaps the MMA of other stages.
//   warp 1        MMA issuer: one thread issues tcgen05.mma kind::f16
//                 (M=128, N=256, K=16): per 16-wide K slice two MMAs, one per
//                 128-row half of the A tile, both reading the same dequantized
//                 weight tile -- so each decoded weight and each byte of
//                 weight traffic through shared memory serves 256 rows of A
//                 (shared-memory bandwidth bounds this kernel).  The two
//                 256-column fp32 accumulators fill TMEM; stages are released
//                 with tcgen05.commit.
//   warps 12..15  epilogue: tcgen05.ld both accumulators, multiply by the
//                 scale, apply the fused epilogue, convert (RNE) and store:
//                 16-bit outputs as 32 x 32 boxes staged in shared memory and
//                 written by TMA (TMEM is free again before the stores land),
//                 otherwise directly with bounds guards.
//   warps 2, 3    idle.
// Pair tiles (the plain FP8 / NVFP4 GEMM with M > 128, W8A8 with M > 128,
// any-K FP8 with M > 256; the grouped GEMMs keep one-CTA tiles):
// a cluster of two CTAs on two SMs shares a tile of 512 A rows (W8A8: 256)
// x 256 weight rows.  Each CTA loads its A rows and 128 weight rows and
// decodes only those; the even CTA's MMA thread issues
// tcgen05.mma.cta_group::2 (M = 256: 128 rows from each CTA's A, N = 256:
// 128 weight rows from each CTA) and each CTA's TMEM receives the sums of
// its own rows.  The weight bytes a CTA moves through shared memory per K
// step halve for the same MMA work; the odd CTA's dequant and epilogue warps
// signal the even CTA's barriers remotely, and the MMA's commits reach both
// CTAs' barriers (multicast).
// W8A8 (Fmt::kInt8): the A tile is int8 too and holds 128 rows.  The page's
// int32 accumulation is kept exact on binary16 MMAs: the dequant warps widen
// both operands' codes exactly to binary16, every product is an integer of
// magnitude at most 2^14, and the MMAs accumulate chunks of at most
// kInt8ChunkSteps K steps (1024 K) in float32, where every partial sum is an
// integer of magnitude at most 2^24 and therefore exact.  At the end of each
// chunk the epilogue warps convert the chunk's sums to int32 and add them to
// a running int32 sum kept in the second TMEM accumulator (the MMAs of the
// next chunk wait for that hand-over); after the tile's last chunk the
// dequant multiplies by a_scale[m] and b_scale[n].  A split-K cluster adds
// its CTAs' int32 partials exactly.
// Tiles are visited m-fastest so that consecutive CTAs share a weight tile
// through L2 (the pages' Morton raster serves the same purpose).
//
// Any K (FP8 only; the "fp4_matmul" page's K-strip plus tail loop): when K is
// not a multiple of 16 the rows of A (2K bytes) and W (K bytes) are not
// 16-byte strided, but rows 8 apart in A (16K bytes) and R = 16 / gcd(K, 16)
// apart in W (RK bytes; R = 2 when K % 16 == 8) are.  So A is described as
// [M/8 groups, 8K elements] and W as [N/R groups, RK bytes]: one TMA box per
// residue class (row mod 8, row mod R) brings the
// 16-byte-aligned windows around the stage's K range of every row of that
// class (rows of an incomplete last group come by cp.async).  The dequant
// warps then shift each row by its fixed misalignment, zero the K tail, and
// write A and the decoded weight in the swizzled layout.  A's rows are
// realigned in place and kept in residue order (tile row 8 i + r at smem row
// 32 r + i), which the epilogue undoes when it picks the output row.  When
// K % 8 == 0, A's rows are 16-byte strided and A comes as the plain tiled
// box of the main path instead (normal row order, no realignment).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gq {
namespace {

constexpr int BM = 256;          // A rows per tile (two MMA halves)
constexpr int UMMA_M = 128;      // rows per tcgen05.mma
constexpr int BN = 256;          // weight rows per tile (MMA N)
constexpr int BK = 64;           // K per stage (one 128-byte swizzle row of bf16)
constexpr int UMMA_K = 16;       // K per tcgen05.mma (kind::f16)
constexpr int kRawStages = 3;
constexpr int kL2Prefetch = 8;   // weight tiles prefetched into L2 this many K steps ahead
constexpr int kDeqStages = 2;
constexpr int kThreads = 512;    // 16 warps
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kDeqWarp0 = 4;
constexpr int kDeqWarps = 8;     // 256 threads: one weight row each
constexpr int kEpiWarp0 = 12;    // 4 warps: TMEM lane groups 0..3
constexpr int kTmemCols = 512;   // two 256-column fp32 accumulators (one per A half; W8A8:
                                 // the chunk's float32 sums and the running int32 sums)

constexpr uint32_t kPartStride = BN * 4 + 16;   // split-K partial row: 256 fp32 + pad
// W8A8: K steps per float32 chunk.  |code| <= 128, so every product is at
// most 2^14 and a chunk's partial sums at most 16 * 64 * 2^14 = 2^24 in
// magnitude: integers that float32 holds exactly.
constexpr int kInt8ChunkSteps = 16;
static_assert(static_cast<int64_t>(kInt8ChunkSteps) * BK * 128 * 128 <= (1LL << 24),
              "W8A8 chunk sums are exact in float32");
static_assert(kInt8MaxK * 128 * 128 < (1LL << 31), "W8A8 int32 sums cannot overflow");
constexpr int kMaxClusterSplit = 8;   // K split over at most a portable cluster
constexpr uint32_t kABytes = BM * BK * 2;        // 32 KB
constexpr uint32_t kAHalfBytes = UMMA_M * BK * 2;  // 16 KB: offset of the second A half
constexpr uint32_t kDeqBytes = BN * BK * 2;      // 32 KB

// kInt8: the W8A8 sibling method (both operands int8, per-row / per-column
// scales), run on the same pipeline with both operands widened to binary16.
enum class Fmt { kFp8, kNvfp4, kInt8 };

template <Fmt F> struct RawLayout;
template <> struct RawLayout<Fmt::kFp8> {
  static constexpr uint32_t kWBytes = BN * BK;          // 16 KB, 64-byte swizzle
  static constexpr uint32_t kScaleBytes = 0;
};
template <> struct RawLayout<Fmt::kNvfp4> {
  static constexpr uint32_t kWBytes = BN * BK / 2;      // 8 KB, 32-byte swizzle
  static constexpr uint32_t kScaleBytes = BN * BK / 16; // 1 KB, 4 bytes per row
};
template <> struct RawLayout<Fmt::kInt8> {
  static constexpr uint32_t kWBytes = BN * BK;          // 16 KB, 64-byte swizzle
  static constexpr uint32_t kScaleBytes = 0;
};

template <Fmt F> struct Smem {
  static constexpr int kRawSt = kRawStages;     // A + raw weight ring
  static constexpr int kDeqSt = kDeqStages;     // decoded weight ring
  static constexpr int kWRows = BN;             // weight rows this CTA loads and decodes
  static constexpr uint32_t kWBytes = RawLayout<F>::kWBytes;
  static constexpr uint32_t kScaleBytes = RawLayout<F>::kScaleBytes;
  static constexpr uint32_t kAStride = kABytes;
  static constexpr uint32_t kARawBytes = kABytes;   // A bytes the TMA brings per stage
  static constexpr bool kADeq = false;              // A read by the MMA from the A ring
  static constexpr uint32_t kDeqAOff = 0;
  static constexpr uint32_t kDeqStride = kDeqBytes;
  static constexpr uint32_t kDeqOff = 0;
  static constexpr uint32_t kAOff = kDeqOff + kDeqStages * kDeqBytes;
  static constexpr uint32_t kWOff = kAOff + kRawStages * kABytes;
  static constexpr uint32_t kSOff = kWOff + kRawStages * RawLayout<F>::kWBytes;
  static constexpr uint32_t kBarOff = (kSOff + kRawStages * RawLayout<F>::kScaleBytes + 7) & ~7u;
  // barriers: full_raw, empty_raw (kRawStages each), full_deq, empty_deq
  // (kDeqStages each), tmem_full, tmem_empty (2 each), drain (1)
  static constexpr uint32_t kNumBars = 2 * kRawStages + 2 * kDeqStages + 4 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;   // tmem addr, abort flag
  // Output staging for TMA stores: 2 buffers of a 32 x 32 16-bit box per
  // epilogue warp (1 KB aligned, 64-byte swizzle).
  static constexpr uint32_t kStageOff = (kMiscOff + 16 + 1023) & ~1023u;
  static constexpr uint32_t kStageBytes = 4 * 2 * 2048;
  static constexpr uint32_t kTotal = kStageOff + kStageBytes;
  static constexpr uint32_t kAlloc = kTotal + 1024;              // slack for 1 KB alignment
};

// Any-K layout: two stages, each [A 32 KB | decoded W 32 KB | A side rows |
// raw W boxes | cp.async rows].  The A box of residue r (rows 8 i + r,
// i < 28; 144 bytes each) lands inside the 4 KB of smem rows 32 r .. 32 r + 31,
// which the same warp overwrites with the realigned rows after reading them;
// the box for i = 28..31 lands in the side area.
constexpr uint32_t kAnyRowA = 144;                 // raw A window bytes per row
constexpr uint32_t kAnyRowW = 80;                  // raw weight window bytes per row
constexpr int kAnyInTile = 28;                     // A box rows that land in place
constexpr uint32_t kAnySideSlot = 640;             // 4 x 144 bytes, rounded to 128
constexpr uint32_t kAnyWArea = BN * kAnyRowW;      // raw W windows of a tile's 256 weight rows
static_assert(kAnyInTile * kAnyRowA <= 32 * BK * 2, "in-place A rows fit their 4 KB");
struct SmemAnyK {
  static constexpr int kRawSt = 2;
  static constexpr int kDeqSt = 2;
  static constexpr int kWRows = BN;
  static constexpr uint32_t kWBytes = RawLayout<Fmt::kFp8>::kWBytes;   // (unused: own boxes)
  static constexpr uint32_t kScaleBytes = 0;
  static constexpr uint32_t kAOff = 0;
  static constexpr uint32_t kDeqOff = kABytes;
  static constexpr uint32_t kSideOff = kABytes + kDeqBytes;
  static constexpr uint32_t kWOff = kSideOff + 8 * kAnySideSlot;
  static constexpr uint32_t kPartAOff = kWOff + kAnyWArea;           // <= 7 rows of A
  static constexpr uint32_t kPartWOff = kPartAOff + 1024;             // <= 15 rows of W
  static constexpr uint32_t kStage = (kPartWOff + 1280 + 1023) & ~1023u;
  static constexpr uint32_t kAStride = kStage;
  static constexpr uint32_t kARawBytes = kABytes;
  static constexpr bool kADeq = false;
  static constexpr uint32_t kDeqAOff = 0;
  static constexpr uint32_t kDeqStride = kStage;
  static constexpr uint32_t kBarOff = 2 * kStage;
  static constexpr uint32_t kNumBars = 2 * kRawStages + 2 * kDeqStages + 4 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStageOff = 0, kStageBytes = 0;   // no TMA-store staging
  static constexpr uint32_t kTotal = kMiscOff + 16;
  static constexpr uint32_t kAlloc = kTotal + 1024;
  // Transaction bytes of one stage's boxes.
  static constexpr uint32_t kABoxBytes = 8 * 32 * kAnyRowA;
  static constexpr uint32_t kWBoxBytes = kAnyWArea;
};

// Pair tiles (cta_group::2): the two CTAs of a cluster pair share a tile of
// kPairBM A rows x BN weight rows.  Each CTA holds 256 A rows (the 128-row
// halves h = 0, 1 are tile rows 256 h + 128 rank + [0, 128)) and loads and
// decodes 128 of the weight rows (tile rows 128 rank + [0, 128)); one thread
// of the even CTA issues M = 256, N = 256 MMAs that read both CTAs' operands,
// and each CTA's TMEM receives the sums of its own A rows.  Per K step a CTA
// moves half the weight bytes through shared memory that a one-CTA tile of
// 256 rows does, for the same MMA work.
constexpr int kPairBM = 512;
constexpr int kPairWRows = BN / 2;
template <Fmt F> struct SmemPair {
  // 3 raw + 3 decoded stages: M = 2048 FP8 143.2 us against 145.4 us with
  // 4 + 2 (3 + 4: 143.9, 3 + 2: 145.9, 2 + 4: 189.6).
  static constexpr int kRawSt = 3;
  static constexpr int kDeqSt = 3;
  static constexpr int kWRows = kPairWRows;
  static constexpr uint32_t kWBytes = RawLayout<F>::kWBytes / 2;
  static constexpr uint32_t kScaleBytes = RawLayout<F>::kScaleBytes / 2;
  static constexpr uint32_t kAStride = kABytes;
  static constexpr uint32_t kARawBytes = kABytes;
  static constexpr bool kADeq = false;
  static constexpr uint32_t kDeqAOff = 0;
  static constexpr uint32_t kDeqStride = kDeqBytes / 2;     // 128 decoded rows
  static constexpr uint32_t kDeqOff = 0;
  static constexpr uint32_t kAOff = kDeqOff + kDeqSt * kDeqStride;
  static constexpr uint32_t kWOff = kAOff + kRawSt * kABytes;
  static constexpr uint32_t kSOff = kWOff + kRawSt * kWBytes;
  static constexpr uint32_t kBarOff = (kSOff + kRawSt * kScaleBytes + 7) & ~7u;
  static constexpr uint32_t kNumBars = 2 * kRawSt + 2 * kDeqSt + 4 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStageOff = (kMiscOff + 16 + 1023) & ~1023u;
  static constexpr uint32_t kStageBytes = 4 * 2 * 2048;
  static constexpr uint32_t kTotal = kStageOff + kStageBytes;
  static constexpr uint32_t kAlloc = kTotal + 1024;
};
// W8A8 pair tiles: 256 output rows (128 per CTA) x 256 weight rows; the
// decoded stage holds the CTA's 128 weight rows and its 128 A rows as
// binary16 (W at +0, A at +16 KB).
template <> struct SmemPair<Fmt::kInt8> {
  static constexpr int kRawSt = 4;
  static constexpr int kDeqSt = 4;
  static constexpr int kWRows = kPairWRows;
  static constexpr uint32_t kWBytes = RawLayout<Fmt::kInt8>::kWBytes / 2;   // 8 KB
  static constexpr uint32_t kScaleBytes = 0;
  static constexpr uint32_t kARawBytes = UMMA_M * BK;                       // 8 KB
  static constexpr uint32_t kAStride = kARawBytes;
  static constexpr bool kADeq = true;
  static constexpr uint32_t kDeqAOff = kDeqBytes / 2;                       // 16 KB
  static constexpr uint32_t kDeqStride = kDeqBytes / 2 + kAHalfBytes;       // 32 KB
  static constexpr uint32_t kDeqOff = 0;
  static constexpr uint32_t kAOff = kDeqOff + kDeqSt * kDeqStride;
  static constexpr uint32_t kWOff = kAOff + kRawSt * kAStride;
  static constexpr uint32_t kSOff = kWOff + kRawSt * kWBytes;
  static constexpr uint32_t kBarOff = kSOff;
  static constexpr uint32_t kNumBars = 2 * kRawSt + 2 * kDeqSt + 4 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStageOff = 0, kStageBytes = 0;   // no TMA-store staging
  static constexpr uint32_t kTotal = kMiscOff + 16;
  static constexpr uint32_t kAlloc = kTotal + 1024;
};
static_assert(SmemPair<Fmt::kFp8>::kAlloc <= 232448 && SmemPair<Fmt::kNvfp4>::kAlloc <= 232448 &&
                  SmemPair<Fmt::kInt8>::kAlloc <= 232448,
              "pair stages and output staging fit in shared memory");

// Any-K pair tiles: each CTA realigns its 256 rows of A (tile rows
// 256 rank + [0, 256), residue order as SmemAnyK) and decodes 128 weight rows
// (one box per W residue class); three stages.
constexpr uint32_t kAnyPairWArea = kPairWRows * kAnyRowW;   // raw W windows of a CTA's 128 rows
struct SmemAnyKPair {
  static constexpr int kRawSt = 3;
  static constexpr int kDeqSt = 3;
  static constexpr int kWRows = kPairWRows;
  static constexpr uint32_t kWBytes = RawLayout<Fmt::kFp8>::kWBytes;   // (unused: own boxes)
  static constexpr uint32_t kScaleBytes = 0;
  static constexpr uint32_t kAOff = 0;
  static constexpr uint32_t kDeqOff = kABytes;
  static constexpr uint32_t kSideOff = kABytes + kDeqBytes / 2;
  static constexpr uint32_t kWOff = kSideOff + 8 * kAnySideSlot;
  static constexpr uint32_t kPartAOff = kWOff + kAnyPairWArea;         // <= 7 rows of A
  static constexpr uint32_t kPartWOff = kPartAOff + 1024;              // <= 15 rows of W
  static constexpr uint32_t kStage = (kPartWOff + 1280 + 1023) & ~1023u;
  static constexpr uint32_t kAStride = kStage;
  static constexpr uint32_t kARawBytes = kABytes;
  static constexpr bool kADeq = false;
  static constexpr uint32_t kDeqAOff = 0;
  static constexpr uint32_t kDeqStride = kStage;
  static constexpr uint32_t kBarOff = kRawSt * kStage;
  static constexpr uint32_t kNumBars = 2 * kRawSt + 2 * kDeqSt + 4 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStageOff = 0, kStageBytes = 0;   // no TMA-store staging
  static constexpr uint32_t kTotal = kMiscOff + 16;
  static constexpr uint32_t kAlloc = kTotal + 1024;
  static constexpr uint32_t kABoxBytes = SmemAnyK::kABoxBytes;
  static constexpr uint32_t kWBoxBytes = kAnyPairWArea;
};
static_assert(SmemAnyKPair::kAlloc <= 232448, "any-K pair stages fit in shared memory");

template <Fmt F, bool kAnyK, bool kPair>
using SmemFor = typename std::conditional<
    kAnyK, typename std::conditional<kPair, SmemAnyKPair, SmemAnyK>::type,
    typename std::conditional<kPair, SmemPair<F>, Smem<F>>::type>::type;

// W8A8: raw int8 A (8 KB, 128 rows) and W (16 KB) stages, 64-byte swizzle,
// and decoded stages holding the weight and A as binary16 (W at +0, A at
// +32 KB).
template <> struct Smem<Fmt::kInt8> {
  static constexpr int kRawSt = kRawStages;
  static constexpr int kDeqSt = 3;
  static constexpr int kWRows = BN;
  static constexpr uint32_t kWBytes = RawLayout<Fmt::kInt8>::kWBytes;
  static constexpr uint32_t kScaleBytes = 0;
  static constexpr uint32_t kARawBytes = UMMA_M * BK;         // 8 KB: 128 rows of int8 A
  static constexpr uint32_t kAStride = kARawBytes;
  static constexpr bool kADeq = true;                         // MMA reads A from the decoded stage
  static constexpr uint32_t kDeqAOff = kDeqBytes;
  static constexpr uint32_t kDeqStride = kDeqBytes + kAHalfBytes;  // 48 KB
  static constexpr uint32_t kDeqOff = 0;
  static constexpr uint32_t kAOff = kDeqOff + kDeqSt * kDeqStride;
  static constexpr uint32_t kWOff = kAOff + kRawStages * kAStride;
  static constexpr uint32_t kSOff = kWOff + kRawStages * RawLayout<Fmt::kInt8>::kWBytes;
  static constexpr uint32_t kBarOff = kSOff;
  static constexpr uint32_t kNumBars = 2 * kRawStages + 2 * kDeqSt + 4 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kStageOff = 0, kStageBytes = 0;   // no TMA-store staging
  static constexpr uint32_t kTotal = kMiscOff + 16;
  static constexpr uint32_t kAlloc = kTotal + 1024;
};
static_assert(Smem<Fmt::kInt8>::kAlloc <= 232448, "W8A8 stages fit in shared memory");
static_assert(Smem<Fmt::kFp8>::kAlloc <= 232448 && Smem<Fmt::kNvfp4>::kAlloc <= 232448,
              "stages and output staging fit in shared memory");

static_assert(UMMA_M * kPartStride <= Smem<Fmt::kInt8>::kBarOff &&
              UMMA_M * kPartStride <= Smem<Fmt::kNvfp4>::kBarOff &&
                  UMMA_M * kPartStride <= Smem<Fmt::kFp8>::kBarOff &&
                  UMMA_M * kPartStride <= SmemAnyK::kBarOff,
              "split-K partials fit below the barriers");
static_assert(SmemAnyK::kAlloc <= 232448, "any-K stages fit in shared memory");

// Work description shared by the plain and grouped GEMMs.
struct Problem {
  void* out;
  const uint32_t* a_offsets;   // grouped only
  const int32_t* expert_ids;   // grouped only
  const float* expert_scales;  // grouped only (may be null)
  uint32_t* status;
  float alpha;
  int M, N, K;                 // M = total rows for grouped
  int bm;                      // A rows per tile (BM; W8A8: UMMA_M; pair tiles: kPairBM)
  int num_n_tiles;
  int num_k_blocks;
  int G, E, max_rows;          // grouped only
  int a_groups, w_groups;      // any-K path: full 8-row groups of A, w_res-row groups of W
  int w_res;                   // any-K path: W rows per 16-byte-strided group, 16 / gcd(K, 16)
  int a_res;                   // any-K path, K % 8 != 0: A rows per group, 8 / gcd(K, 8)
  int tma_out;                 // 16-bit output stored through the output tensor map
  int a_tma;                   // any-K path with K % 8 == 0: A by the plain tiled map
  Epi ep;                      // output type and fused epilogue
  const float* a_scale;        // W8A8: per-row scale of A [M]
  const float* b_scale;        // W8A8: per-output-column scale of W [N]
  const void* a_g;             // any-K path: A [M, K] bf16
  const uint8_t* w_g;          // any-K path: W [N, K] e4m3 codes
  int ksplit;                  // > 1: split-K over a thread-block cluster of ksplit CTAs
  int kb_per_split;            // K steps per split
  int stall_producer;          // GQ_LAUNCH_TEST_STALL_PRODUCER: the producer issues nothing
};

// A tile of work: rows [m0, m_end) of C, columns [n0, n0 + BN), weight index.
struct Tile {
  int m0, m_end, n0, expert;  // expert: -1 = write zeros, >= 0 = weight matrix index
  float scale;
  bool valid;
};

// Plain GEMM: tile t -> (m tile fastest, n tile).
__device__ __forceinline__ Tile plain_tile(const Problem& p, int t) {
  const int num_m = (p.M + p.bm - 1) / p.bm;
  Tile tl;
  tl.m0 = (t % num_m) * p.bm;
  tl.m_end = min(tl.m0 + p.bm, p.M);
  tl.n0 = (t / num_m) * BN;
  tl.expert = 0;
  tl.scale = p.alpha;
  tl.valid = true;
  return tl;
}

__device__ __forceinline__ int plain_num_tiles(const Problem& p) {
  return ((p.M + p.bm - 1) / p.bm) * p.num_n_tiles;
}

// Grouped GEMM: the work list is every (group, m tile, n tile) whose group has
// rows, enumerated group by group, n tile, then m tile (fastest).  Each role
// derives it from a_offsets / expert_ids (read-only device data) by a scan over
// the groups, so no host synchronization and no scratch memory are needed.
__device__ __forceinline__ int group_rows(const Problem& p, int z, int* start) {
  int s = static_cast<int>(min(__ldg(p.a_offsets + z), static_cast<uint32_t>(p.M)));
  int e = static_cast<int>(min(__ldg(p.a_offsets + z + 1), static_cast<uint32_t>(p.M)));
  *start = s;
  int rows = e > s ? e - s : 0;
  return min(rows, p.max_rows);
}

__device__ __forceinline__ int grouped_num_tiles(const Problem& p) {
  int total = 0;
  for (int z = 0; z < p.G; ++z) {
    int s;
    const int rows = group_rows(p, z, &s);
    total += ((rows + p.bm - 1) / p.bm) * p.num_n_tiles;
  }
  return total;
}

__device__ __forceinline__ Tile grouped_tile(const Problem& p, int t) {
  Tile tl;
  tl.valid = false;
  for (int z = 0; z < p.G; ++z) {
    int s;
    const int rows = group_rows(p, z, &s);
    const int mt = (rows + p.bm - 1) / p.bm;
    const int cnt = mt * p.num_n_tiles;
    if (t < cnt) {
      tl.m0 = s + (t % mt) * p.bm;
      tl.m_end = min(tl.m0 + p.bm, s + rows);
      tl.n0 = (t / mt) * BN;
      const int id = __ldg(p.expert_ids + z);
      tl.expert = (id >= 0 && id < p.E) ? id : -1;
      tl.scale = (tl.expert >= 0 && p.expert_scales != nullptr) ? __ldg(p.expert_scales + tl.expert)
                                                                   : 1.0f;
      tl.valid = true;
      return tl;
    }
    t -= cnt;
  }
  return tl;
}

template <bool kGrouped>
__device__ __forceinline__ Tile get_tile(const Problem& p, int t) {
  if constexpr (kGrouped) return grouped_tile(p, t);
  else return plain_tile(p, t);
}

template <bool kGrouped>
__device__ __forceinline__ int num_tiles(const Problem& p) {
  if constexpr (kGrouped) return grouped_num_tiles(p);
  else return plain_num_tiles(p);
}

// ------------------------------------------------------ any-K loading --

// A CTA's 256 rows of A in R residue classes (rows R i + r, R = 2, 4 or 8):
// rr = 256 / R rows per class, whose realigned rows occupy smem rows
// rr r .. rr r + rr - 1 (128 rr bytes).  The first ip = floor(128 rr / 144)
// raw windows of class r land in place inside those bytes, the other
// rr - ip in the class's side slot (rounded up to 128 bytes).
__host__ __device__ constexpr int any_a_in_place(int R) { return (256 / R) * 128 / static_cast<int>(kAnyRowA); }
__host__ __device__ constexpr uint32_t any_a_side_slot(int R) {
  return ((static_cast<uint32_t>(256 / R - any_a_in_place(R)) * kAnyRowA + 127u) / 128u) * 128u;
}
static_assert(any_a_in_place(8) == kAnyInTile && any_a_side_slot(8) == kAnySideSlot,
              "eight classes: 28 rows in place, 4 in a 640-byte slot");
static_assert(2 * any_a_side_slot(2) <= 8 * kAnySideSlot && 4 * any_a_side_slot(4) <= 8 * kAnySideSlot,
              "the side slots of every class count fit the side area");

// Where the raw window of class r (of R), group index i (tile row R i + r) of
// a stage lands, relative to the stage (side_off: the layout's side area).
__device__ __forceinline__ uint32_t any_raw_a_off(int R, int r, int i, uint32_t side_off) {
  const int ip = any_a_in_place(R);
  return i < ip ? static_cast<uint32_t>(r * (256 / R) * 128 + i * kAnyRowA)
                : side_off + r * any_a_side_slot(R) + (i - ip) * kAnyRowA;
}

// The bytes [off, off + 4 N) of in[] (off = 0..15, a per-row constant), as
// N words: a two-step word shift by off / 4 and a funnel shift by off % 4,
// with constant register indices.
template <int N>
__device__ __forceinline__ void realign_words(const uint32_t (&in)[N + 4], uint32_t off,
                                              uint32_t (&out)[N]) {
  const bool s2 = off & 8, s1 = off & 4;
  const uint32_t sh = (off & 3) * 8;
  uint32_t t[N + 2], u[N + 1];
#pragma unroll
  for (int i = 0; i < N + 2; ++i) t[i] = s2 ? in[i + 2] : in[i];
#pragma unroll
  for (int i = 0; i < N + 1; ++i) u[i] = s1 ? t[i + 1] : t[i];
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(u[i], u[i + 1], sh);
}

// Zero the bytes at or after nbytes (the K tail of the last stage).
template <int N>
__device__ __forceinline__ void mask_tail(uint32_t (&w)[N], int nbytes) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int rem = nbytes - 4 * i;
    const uint32_t m = rem >= 4 ? 0xFFFFFFFFu : rem <= 0 ? 0u : (1u << (8 * rem)) - 1u;
    w[i] &= m;
  }
}

// Prefetch the bytes [lo, hi) of a buffer that starts 16-byte aligned at
// `base` into L2, in 32 KB pieces spread over the lanes of a warp; the range
// is shrunk to 16-byte boundaries inside [base, hi).
__device__ __forceinline__ void prefetch_span_l2(const uint8_t* base, int64_t lo, int64_t hi,
                                                 int lane) {
  lo &= ~static_cast<int64_t>(15);
  hi &= ~static_cast<int64_t>(15);
  constexpr int64_t kPiece = 32768;
  for (int64_t o = lo + lane * kPiece; o < hi; o += 32 * kPiece)
    tc::bulk_prefetch_l2(base + o, static_cast<uint32_t>(min(kPiece, hi - o)));
}

// W8A8: a chunk's float32 sum (an exact integer of magnitude <= 2^24, so the
// conversion is exact) plus the running int32 sum of the earlier chunks.
__device__ __forceinline__ int chunk_sum(uint32_t chunk_bits, uint32_t run_bits, bool have_run) {
  return __float2int_rz(__uint_as_float(chunk_bits)) + (have_run ? static_cast<int>(run_bits) : 0);
}

// ----------------------------------------------------------------- kernel --

template <Fmt F, bool kGrouped, bool kAnyK, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
k_wq_gemm(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
          const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_o,
          const uint8_t* __restrict__ scales_g, Problem p) {
  static_assert(!kPair || !kAnyK || (F == Fmt::kFp8 && !kGrouped), "any-K pair tiles: plain FP8");
  using L = SmemFor<F, kAnyK, kPair>;
  // The any-K roles' layout (the same type as L when kAnyK; the roles are
  // compiled, never run, in the other instantiations).
  using LA = typename std::conditional<kPair, SmemAnyKPair, SmemAnyK>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full_raw = bars;
  uint64_t* empty_raw = bars + L::kRawSt;
  uint64_t* full_deq = bars + 2 * L::kRawSt;
  uint64_t* empty_deq = full_deq + L::kDeqSt;
  uint64_t* tmem_full = empty_deq + L::kDeqSt;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = tc::smem_u32(smem);
  // Pair tiles: rank 0 of the pair issues the MMAs; the other roles run in
  // both CTAs on the CTA's own rows.
  const int prank = kPair ? static_cast<int>(tc::cluster_ctarank()) : 0;

  if (threadIdx.x == 0) {
    // The raw stage is full after the copies (+ the NVFP4 scale copies).  It
    // is empty after the MMA (+ the dequant warps that read its raw weight;
    // any K: the loader warps finish with a stage before the MMA starts;
    // W8A8: the MMA reads only decoded stages, so the dequant warps alone).
    constexpr uint32_t kRawArrivals = (kAnyK || F == Fmt::kNvfp4) ? 1 + 32 : 1;
    constexpr uint32_t kRawReleases = kAnyK ? 1 : F == Fmt::kInt8 ? kDeqWarps : 1 + kDeqWarps;
    // Pair tiles: the even CTA's full_deq and tmem_empty also count the odd
    // CTA's dequant and epilogue warps (remote arrivals); the MMA's commits
    // reach the barriers of both CTAs.
    for (int s = 0; s < L::kRawSt; ++s) {
      tc::mbar_init(&full_raw[s], kRawArrivals);
      tc::mbar_init(&empty_raw[s], kRawReleases);
    }
    for (int s = 0; s < L::kDeqSt; ++s) {
      tc::mbar_init(&full_deq[s], kPair ? 2 * kDeqWarps : kDeqWarps);
      tc::mbar_init(&empty_deq[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&tmem_full[s], 1);
      tc::mbar_init(&tmem_empty[s], kPair ? 8 : 4);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    if constexpr (kPair) {
      tc::tmem_alloc_pair(tmem_slot, kTmemCols);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(tmem_slot, kTmemCols);
      tc::tmem_relinquish();
    }
  }
  if (!kAnyK && warp == kWarpTma && lane == 0 && p.num_k_blocks > 0 && (!kGrouped || p.E > 0)) {
    tc::tma_prefetch_desc(&tmap_a);
    tc::tma_prefetch_desc(&tmap_w);
  }
  if (kAnyK && warp == kWarpTma && lane == 0) {
    if (p.a_tma) tc::tma_prefetch_desc(&tmap_a);
    if (p.a_groups > 0) {
      tc::tma_prefetch_desc(&tmap_a);
      tc::tma_prefetch_desc(&tmap_x);
    }
    if (p.w_groups > 0) tc::tma_prefetch_desc(&tmap_w);
  }
  tc::tc_fence_before();
  // Pair tiles: the peer's barriers are initialized before any remote arrival
  // or multicast commit can reach them.
  if constexpr (kPair) tc::cluster_sync();
  else __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_tiles = num_tiles<kGrouped>(p);
  // Split-K (small M): the CTAs of a cluster share one tile, rank r owns the
  // K steps [kb0, kb1); otherwise a CTA walks tiles persistently over all K.
  // Pair tiles: the pair (cluster) walks the tiles persistently.
  const bool split = p.ksplit > 1;
  const int crank = split ? static_cast<int>(blockIdx.x) % p.ksplit : 0;
  const int unit = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  const int t_first = split ? static_cast<int>(blockIdx.x) / p.ksplit : unit;
  const int t_step = split ? total_tiles : units;
  // Pair tiles: this CTA's first weight row within the tile's BN rows, and
  // the offset of its A rows within each 256-row half of the tile.
  const int w_row0 = kPair ? prank * kPairWRows : 0;
  const int a_row0 = kPair ? prank * (kAnyK ? BM : UMMA_M) : 0;
  // (W8A8: one MMA half of 128 rows per CTA; the second accumulator holds
  // the running int32 sums.  Any K: CTA r holds tile rows 256 r + [0, 256)
  // -- in residue order, or in order as halves of 128 -- and both halves are
  // always issued.)
  constexpr int kHalfRows = (kPair && F != Fmt::kInt8 && !kAnyK) ? 2 * UMMA_M : UMMA_M;   // tile rows per MMA half
  const int kb0 = split ? crank * p.kb_per_split : 0;
  const int kb1 = split ? min(p.num_k_blocks, kb0 + p.kb_per_split) : p.num_k_blocks;
  const int nkb = kb1;

  if (warp == kWarpTma && p.stall_producer) {
    // Failure-path test: no copy is issued, so every stage stays empty and
    // the other roles' bounded waits run out (nothing asynchronous to drain).
  } else if (warp == kWarpTma && !kAnyK) {
    // ------------------------------------------------------ TMA producer --
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    // Weight tiles are prefetched into L2 kL2Prefetch K steps ahead (into the
    // CTA's next tile near the end of a tile): the ring holds only a few
    // stages, too few to hide DRAM latency when the weight is not yet in L2
    // (grouped: every expert's weight streams from DRAM once).
    auto prefetch_w = [&](const Tile& pt, int pkb) {
      if (lane != 0 || !pt.valid || pt.expert < 0) return;
      constexpr int kBpk = (F == Fmt::kNvfp4) ? BK / 2 : BK;   // weight bytes per row per K step
      if constexpr (kGrouped) tc::tma_prefetch_l2_3d(&tmap_w, pkb * kBpk, pt.n0 + w_row0, pt.expert);
      else tc::tma_prefetch_l2_2d(&tmap_w, pkb * kBpk, pt.n0 + w_row0);
    };
    if (t_first < total_tiles) {
      const Tile first = get_tile<kGrouped>(p, t_first);
      for (int kb = kb0; kb < kb0 + kL2Prefetch && kb < nkb; ++kb) prefetch_w(first, kb);
    }
    for (int t = t_first; t < total_tiles && ok; t += t_step) {
      const Tile tl = get_tile<kGrouped>(p, t);
      if (!tl.valid || tl.expert < 0) continue;
      const int tn = t + t_step;
      Tile next{};
      next.valid = false;
      if (tn < total_tiles) next = get_tile<kGrouped>(p, tn);
      // Pair tiles: the second 128-row half of this CTA's A rows only when
      // the tile has more than 256 rows.
      const int a_halves = (kPair && tl.m_end - tl.m0 <= kHalfRows) ? 1 : 2;
      for (int kb = kb0; kb < nkb; ++kb) {
        if (kb + kL2Prefetch < nkb) prefetch_w(tl, kb + kL2Prefetch);
        else if (kb + kL2Prefetch - nkb < nkb && !split) prefetch_w(next, kb + kL2Prefetch - nkb);
        if (!tc::mbar_wait<kPair>(&empty_raw[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* a_dst = smem + L::kAOff + s * L::kAStride;
        uint8_t* w_dst = smem + L::kWOff + s * L::kWBytes;
        if (lane == 0) {
          if constexpr (kPair && F == Fmt::kInt8) {
            tc::mbar_arrive_expect_tx(&full_raw[s], L::kARawBytes + L::kWBytes);
            tc::tma_load_2d(a_dst, &tmap_a, &full_raw[s], kb * BK, tl.m0 + a_row0);
          } else if constexpr (kPair) {
            tc::mbar_arrive_expect_tx(&full_raw[s], a_halves * kAHalfBytes + L::kWBytes);
            for (int h = 0; h < a_halves; ++h)
              tc::tma_load_2d(a_dst + h * kAHalfBytes, &tmap_a, &full_raw[s], kb * BK,
                              tl.m0 + h * kHalfRows + a_row0);
          } else {
            tc::mbar_arrive_expect_tx(&full_raw[s], L::kARawBytes + L::kWBytes);
            tc::tma_load_2d(a_dst, &tmap_a, &full_raw[s], kb * BK, tl.m0);
          }
          constexpr int kBpk = (F == Fmt::kNvfp4) ? BK / 2 : BK;
          if constexpr (kGrouped)
            tc::tma_load_3d(w_dst, &tmap_w, &full_raw[s], kb * kBpk, tl.n0 + w_row0, tl.expert);
          else tc::tma_load_2d(w_dst, &tmap_w, &full_raw[s], kb * kBpk, tl.n0 + w_row0);
        }
        if constexpr (F == Fmt::kNvfp4) {
          // Block scales: 4 bytes (4 blocks of 16) per weight row per stage;
          // grouped: rows of expert e start at e * N.
          uint8_t* s_dst = smem + L::kSOff + s * L::kScaleBytes;
          const int ks = p.K / 16;
          const int64_t row_base = kGrouped ? static_cast<int64_t>(tl.expert) * p.N : 0;
#pragma unroll
          for (int i = 0; i < L::kWRows / 32; ++i) {
            const int r = lane + 32 * i;
            const int n = tl.n0 + w_row0 + r;
            const bool in = n < p.N;
            const uint8_t* src = scales_g + ((row_base + (in ? n : 0)) * ks + kb * 4);
            tc::cp_async_4(s_dst + r * 4, src, in ? 4u : 0u);
          }
          tc::cp_async_mbar_arrive_noinc(&full_raw[s]);
        }
        if (++s == L::kRawSt) { s = 0; ph ^= 1; }
      }
    }
    // Drain: make sure no copy issued by this warp is still landing in shared
    // memory when the CTA exits (bounded; normally already complete).
    if (lane == 0) {
      int ds = s;
      uint32_t dph = ph;
      for (int i = 0; i < L::kRawSt; ++i) {
        if (--ds < 0) { ds = L::kRawSt - 1; dph ^= 1; }
        tc::mbar_wait_quiet(&full_raw[ds], dph, 100000000ull);
      }
    }
  } else if (kAnyK && warp == kWarpTma) {
    // ------------------------------------------------ any-K TMA producer --
    // Per stage, lanes 0 .. 2 R_A - 1: R_A + R_A A boxes (class r: rows
    // R_A i + r, i < ip and i >= ip); lanes 16 .. 16 + R_W - 1: the R_W W boxes
    // (class r: rows R_W i + r), each box starting at the stage's K offset of
    // its class rounded down to 16 bytes.  All lanes: the rows past the last full group by 16-byte
    // cp.async (a chunk that crosses the end of its buffer copies only the
    // bytes inside it).
    const uint8_t* a_g = static_cast<const uint8_t*>(p.a_g);
    const int64_t K = p.K;
    const uint8_t* a_end = a_g + 2 * static_cast<int64_t>(p.M) * K;
    const uint8_t* w_end = p.w_g + static_cast<int64_t>(p.N) * K;
    const int a_full = p.a_res * p.a_groups;      // rows covered by the A maps
    const int w_full = p.w_res * p.w_groups;      // rows covered by the W map
    // This CTA's rows of a tile (pair tiles: 256 A rows and 128 weight rows).
    auto cta_rows = [&](const Tile& tt, int& m0c, int& m1c, int& n0c, int& n1c) {
      m0c = tt.m0 + a_row0;
      m1c = min(m0c + BM, tt.m_end);
      n0c = tt.n0 + w_row0;
      n1c = min(n0c + LA::kWRows, p.N);
    };
    auto prefetch_tile = [&](int pt_i) {
      if (pt_i >= total_tiles) return;
      const Tile pt = get_tile<kGrouped>(p, pt_i);
      if (!pt.valid || pt.expert < 0) return;
      int m0c, m1c, n0c, n1c;
      cta_rows(pt, m0c, m1c, n0c, n1c);
      if (n1c > n0c) prefetch_span_l2(p.w_g, n0c * K + kb0 * BK, static_cast<int64_t>(n1c) * K, lane);
      if (m1c > m0c) prefetch_span_l2(a_g, 2 * (m0c * K + kb0 * BK), 2 * static_cast<int64_t>(m1c) * K, lane);
    };
    // One 16-byte chunk at the 16-byte-aligned address src; `any` is a valid
    // address passed when no byte is read.
    auto copy_chunk = [&](uint8_t* dst, const uint8_t* src, const uint8_t* end, const uint8_t* any) {
      const int64_t left = end - src;
      const uint32_t n = left >= 16 ? 16u : left > 0 ? static_cast<uint32_t>(left) : 0u;
      tc::cp_async_16(dst, n ? src : any, n);
    };
    constexpr uint32_t kTx0 = LA::kABoxBytes, kTx1 = LA::kWBoxBytes;
    const uint32_t w_box = static_cast<uint32_t>(LA::kWRows / p.w_res) * kAnyRowW;   // one residue's W box
    // K % 8 == 0: A's rows are 16-byte strided and come as one plain tiled
    // box per stage (128-byte swizzle, the MMA's layout); only W needs the
    // residue boxes.
    const uint32_t tx = (p.a_tma ? kABytes : p.a_groups > 0 ? kTx0 : 0u) + (p.w_groups > 0 ? kTx1 : 0u);
    prefetch_tile(t_first);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = t_first; t < total_tiles && ok; t += t_step) {
      const Tile tl = get_tile<kGrouped>(p, t);
      prefetch_tile(t + t_step);
      if (!tl.valid || tl.expert < 0) continue;
      int m0c, m1c, n0c, n1c;
      cta_rows(tl, m0c, m1c, n0c, n1c);
      const bool a_part = !p.a_tma && m1c > a_full;
      const bool w_part = n1c > w_full;
      for (int kb = kb0; kb < nkb; ++kb) {
        if (!tc::mbar_wait<kPair>(&empty_raw[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) {
          ok = false;
          break;
        }
        const int64_t k0 = static_cast<int64_t>(kb) * BK;
        uint8_t* st = smem + s * LA::kStage;
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(&full_raw[s], tx);
          if (p.a_tma) {
            tc::tma_load_2d(st, &tmap_a, &full_raw[s], static_cast<int>(k0), m0c);
          }
        }
        __syncwarp();   // the stage's expected bytes are set before the other boxes go out
        // A (K % 8 != 0): the two boxes of class r (rows R i + r, i < ip and
        // i >= ip) from lanes r and R + r; W: one box per class (rows
        // w_res i + r) from lane 16 + r -- all issued in parallel.
        if (!p.a_tma && p.a_groups > 0 && lane < 2 * p.a_res) {
          const int R = p.a_res;
          const int r = lane & (R - 1);
          const int x0 = static_cast<int>((r * K + k0) & ~static_cast<int64_t>(7));
          if (lane < R) tc::tma_load_2d(st + any_raw_a_off(R, r, 0, LA::kSideOff), &tmap_a, &full_raw[s], x0, m0c / R);
          else tc::tma_load_2d(st + any_raw_a_off(R, r, any_a_in_place(R), LA::kSideOff), &tmap_x, &full_raw[s],
                               x0, m0c / R + any_a_in_place(R));
        }
        if (p.w_groups > 0 && lane >= 16 && lane < 16 + p.w_res) {
          const int r = lane - 16;
          const int x0 = static_cast<int>((r * K + k0) & ~static_cast<int64_t>(15));
          tc::tma_load_2d(st + LA::kWOff + r * w_box, &tmap_w, &full_raw[s], x0, n0c / p.w_res);
        }
        if (a_part) {
          for (int c = lane; c < 7 * 9; c += 32) {
            const int r = c / 9, j = c - 9 * r;
            const int m = a_full + r;
            if (m < m0c || m >= m1c) continue;
            const uintptr_t w0 = reinterpret_cast<uintptr_t>(a_g + 2 * (m * K + k0)) & ~static_cast<uintptr_t>(15);
            copy_chunk(st + LA::kPartAOff + r * kAnyRowA + 16 * j,
                       reinterpret_cast<const uint8_t*>(w0) + 16 * j, a_end, a_g);
          }
        }
        if (w_part) {
          for (int c = lane; c < 15 * 5; c += 32) {
            const int r = c / 5, j = c - 5 * r;
            const int n = w_full + r;
            if (n < n0c || n >= n1c) continue;
            const uintptr_t w0 = reinterpret_cast<uintptr_t>(p.w_g + n * K + k0) & ~static_cast<uintptr_t>(15);
            copy_chunk(st + LA::kPartWOff + r * kAnyRowW + 16 * j,
                       reinterpret_cast<const uint8_t*>(w0) + 16 * j, w_end, p.w_g);
          }
        }
        tc::cp_async_mbar_arrive_noinc(&full_raw[s]);
        if (++s == LA::kRawSt) { s = 0; ph ^= 1; }
      }
    }
    // Drain: no copy may still land when the CTA exits.
    if (lane == 0) {
      int ds = s;
      uint32_t dph = ph;
      for (int i = 0; i < LA::kRawSt; ++i) {
        if (--ds < 0) { ds = LA::kRawSt - 1; dph ^= 1; }
        tc::mbar_wait_quiet(&full_raw[ds], dph, 100000000ull);
      }
    }
  } else if (warp == kWarpMma && prank == 0) {
    // ------------------------------------------------------- MMA issuer --
    // Pair tiles: M = 256 MMAs over both CTAs' operands, from rank 0 only.
    constexpr int kMmaM = kPair ? 2 * UMMA_M : UMMA_M;
    constexpr uint32_t kIdesc =
        F == Fmt::kInt8 ? tc::idesc_f16_f32(kMmaM, BN) : tc::idesc_bf16_f32(kMmaM, BN);
    // Hand-overs of the accumulators to the epilogue: one per tile (W8A8:
    // one per chunk of at most kInt8ChunkSteps K steps, whose first MMA
    // starts a fresh float32 sum).
    constexpr int kChunk = F == Fmt::kInt8 ? kInt8ChunkSteps : (1 << 30);
    int s = 0, d = 0;
    uint32_t ph = 0, dph = 0;
    int hand = 0;
    bool ok = true;
    for (int t = t_first; t < total_tiles && ok; t += t_step) {
      const Tile tl = get_tile<kGrouped>(p, t);
      if (!tl.valid || tl.expert < 0) continue;
      // (Any K: the rows are in residue order, spread over both halves.)
      // (W8A8: one MMA per K slice; the second accumulator is the epilogue's.)
      const bool two_halves =
          F != Fmt::kInt8 && ((kAnyK && !p.a_tma) || tl.m_end - tl.m0 > kHalfRows);
      for (int cb = kb0; cb < nkb && ok; cb += kChunk) {
        const int ce = nkb - cb > kChunk ? cb + kChunk : nkb;
        // The accumulators are free: the epilogue has read the previous hand-over.
        if (!tc::mbar_wait<kPair>(&tmem_empty[0], (hand & 1) ^ 1, abort_flag, p.status, kStatusTimeoutMma)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        for (int kb = cb; kb < ce; ++kb) {
          // (W8A8: both operands come from the decoded stage; the raw ring is
          // the dequant warps' alone and may run ahead of the MMAs.)
          if ((F != Fmt::kInt8 && !tc::mbar_wait(&full_raw[s], ph, abort_flag, p.status, kStatusTimeoutMma)) ||
              !tc::mbar_wait<kPair>(&full_deq[d], dph, abort_flag, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          if (lane == 0) {
            const uint32_t a_addr = L::kADeq ? smem_base + L::kDeqOff + d * L::kDeqStride + L::kDeqAOff
                                             : smem_base + L::kAOff + s * L::kAStride;
            const uint32_t b_addr = smem_base + L::kDeqOff + d * L::kDeqStride;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              const uint64_t bd = tc::sw128_kmajor_desc(b_addr + kk * UMMA_K * 2);
              const uint64_t a0 = tc::sw128_kmajor_desc(a_addr + kk * UMMA_K * 2);
              const uint64_t a1 = tc::sw128_kmajor_desc(a_addr + kAHalfBytes + kk * UMMA_K * 2);
              const uint32_t accum = (kb > cb || kk > 0) ? 1u : 0u;
              // A tile with at most 128 rows (pair tiles: 256; the ragged end
              // of M or of a group) needs only the first half; the second
              // accumulator is unused.
              if constexpr (kPair) {
                tc::mma_bf16_pair(tmem_base, a0, bd, kIdesc, accum);
                if (two_halves) tc::mma_bf16_pair(tmem_base + BN, a1, bd, kIdesc, accum);
              } else {
                tc::mma_bf16(tmem_base, a0, bd, kIdesc, accum);
                if (two_halves) tc::mma_bf16(tmem_base + BN, a1, bd, kIdesc, accum);
              }
            }
            if constexpr (kPair) {
              if constexpr (F != Fmt::kInt8) tc::mma_commit_pair(&empty_raw[s], 3);
              tc::mma_commit_pair(&empty_deq[d], 3);
            } else {
              if constexpr (F != Fmt::kInt8) tc::mma_commit(&empty_raw[s]);
              tc::mma_commit(&empty_deq[d]);
            }
          }
          __syncwarp();
          if (++s == L::kRawSt) { s = 0; ph ^= 1; }
          if (++d == L::kDeqSt) { d = 0; dph ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) {
          if constexpr (kPair) tc::mma_commit_pair(&tmem_full[0], 3);
          else tc::mma_commit(&tmem_full[0]);
        }
        __syncwarp();
        ++hand;
      }
    }
    // Drain: every MMA issued by this thread completes before TMEM is freed.
    if (lane == 0) {
      if constexpr (kPair) tc::mma_commit_pair(drain, 1);
      else tc::mma_commit(drain);
      tc::mbar_wait_quiet(drain, 0, 100000000ull);
    }
    __syncwarp();
  } else if (kAnyK && warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // ----------------------------------------- any-K realign + dequant --
    // Thread t owns smem A row t (residue t / 32, group index t % 32) and one
    // weight row chosen so that the 8 threads of each quarter warp read
    // distinct 16-byte bank groups of the raw boxes and write distinct ones of
    // the swizzled tile: with R = w_res residues, thread u takes residue
    // u mod R and group index (u / R + rot) mod (rows / R), rot = (u mod R)
    // mod 8 for R >= 8, else (u mod R) * 8 / R -- so that the rows' positions
    // in the raw area differ mod 8 within every quarter warp.  Each raw window
    // is shifted by its fixed misalignment, the K tail of the last stage is
    // zeroed, and rows past the end are zero.  Pair tiles (128 weight rows
    // per CTA): threads t and t + 128 share a weight row, each realigning and
    // decoding half of it.
    constexpr int kWParts = kDeqWarps * 32 / LA::kWRows;   // threads per weight row
    constexpr int kWWords = 16 / kWParts;                  // code words per thread
    const int wres = p.w_res;
    const int wlog = __ffs(wres) - 1;
    const uint32_t w_box = static_cast<uint32_t>(LA::kWRows >> wlog) * kAnyRowW;
    const int t = threadIdx.x - kDeqWarp0 * 32;
    const int ares = p.a_res;                         // A classes (K % 8 != 0)
    const int arlog = 8 - (__ffs(ares) - 1);          // log2 of the rows per class, 256 / ares
    const int ar = t >> arlog, ai = t & ((1 << arlog) - 1);   // A class, group index
    const int u = t % LA::kWRows, wpart = t / LA::kWRows;
    const int wr = u & (wres - 1);                    // W residue
    const int rot = wres >= 8 ? (wr & 7) : (wr << (3 - wlog));
    const int wi = ((u >> wlog) + rot) & ((LA::kWRows >> wlog) - 1);   // W group index
    const int wrow = (wi << wlog) + wr;               // W row in the CTA's part of the tile
    const int64_t K = p.K;
    const int a_full = ares * p.a_groups;
    const int w_full = wres * p.w_groups;
    const uint32_t off_a = static_cast<uint32_t>((2 * ar * K) & 15);
    const uint32_t off_w = static_cast<uint32_t>((wr * K) & 15);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tt = t_first; tt < total_tiles && ok; tt += t_step) {
      const Tile tl = get_tile<kGrouped>(p, tt);
      if (!tl.valid || tl.expert < 0) continue;
      const int m0c = tl.m0 + a_row0;                 // this CTA's rows of the tile
      const int m = m0c + ares * ai + ar;
      const bool a_act = m < min(m0c + BM, tl.m_end);
      const uint32_t a_src = m < a_full ? any_raw_a_off(ares, ar, ai, LA::kSideOff)
                                        : LA::kPartAOff + (m - a_full) * kAnyRowA;
      const int n = tl.n0 + w_row0 + wrow;
      const bool w_act = n < p.N;
      const uint32_t w_src = (n < w_full ? LA::kWOff + wr * w_box + wi * kAnyRowW
                                         : LA::kPartWOff + (n - w_full) * kAnyRowW) +
                             32 * wpart;
      for (int kb = kb0; kb < nkb; ++kb) {
        const bool got = tc::mbar_wait(&full_raw[s], ph, abort_flag, p.status, kStatusTimeoutDequant);
        // With fewer than eight A classes the dequant warps meet at a named
        // barrier each stage, so a failed wait is voted there and every
        // participant leaves together; otherwise each thread leaves at once.
        if (!got && (p.a_tma || ares == 8)) {
          ok = false;
          break;
        }
        const int kv = min(BK, p.K - kb * BK);     // valid K of this stage, >= 1
        const uint32_t st = smem_base + s * LA::kStage;
        if (!p.a_tma) {
          uint32_t out[32];
          if (got && a_act) {
            uint32_t in[36];
#pragma unroll
            for (int c = 0; c < 9; ++c) {
              const uint4 v = tc::lds128(st + a_src + 16 * c);
              in[4 * c] = v.x; in[4 * c + 1] = v.y; in[4 * c + 2] = v.z; in[4 * c + 3] = v.w;
            }
            realign_words<32>(in, off_a, out);
            if (kv < BK) mask_tail<32>(out, 2 * kv);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) out[i] = 0u;
          }
          // Every raw row is read before a realigned row overwrites it: the
          // warp's own rows with eight classes (one warp per class), all
          // dequant warps' with fewer (a class spans several warps).
          if (ares == 8) {
            __syncwarp();
          } else if (tc::bar_red_or<1, kDeqWarps * 32>(!got)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c)
            tc::sts128(st + sw128_off(t, c),
                       make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]));
        }
        {
          // This thread's kWWords code words of its row: bytes
          // [32 wpart, 32 wpart + 4 kWWords) of the stage's 64.
          constexpr uint16_t kOne = 0x3C00;         // 1.0 in f16
          uint32_t code[kWWords];
          if (w_act) {
            uint32_t in[kWWords + 4];
#pragma unroll
            for (int c = 0; c < kWWords / 4 + 1; ++c) {
              const uint4 v = tc::lds128(st + w_src + 16 * c);
              in[4 * c] = v.x; in[4 * c + 1] = v.y; in[4 * c + 2] = v.z; in[4 * c + 3] = v.w;
            }
            realign_words<kWWords>(in, off_w, code);
            if (kv < BK) mask_tail<kWWords>(code, kv - 32 * wpart);
          } else {
#pragma unroll
            for (int i = 0; i < kWWords; ++i) code[i] = 0u;
          }
          const uint32_t dst = st + LA::kDeqOff;
#pragma unroll
          for (int i = 0; i < kWWords / 2; ++i) {
            const int c = (kWWords / 2) * wpart + i;   // 16-byte chunk of the bf16 row
            uint32_t h0, h1, h2, h3;
            e4m3x4_to_h2x2(code[2 * i], h0, h1);
            e4m3x4_to_h2x2(code[2 * i + 1], h2, h3);
            tc::sts128(dst + sw128_off(wrow, c),
                       make_uint4(f32x2_hi_to_bf16x2(h2_scale_f32(h0, kOne)),
                                  f32x2_hi_to_bf16x2(h2_scale_f32(h1, kOne)),
                                  f32x2_hi_to_bf16x2(h2_scale_f32(h2, kOne)),
                                  f32x2_hi_to_bf16x2(h2_scale_f32(h3, kOne))));
          }
        }
        tc::fence_proxy_async_smem();   // make the generic stores visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          // Pair tiles: the MMA issuer (rank 0) waits for both CTAs' rows.
          if constexpr (kPair) tc::mbar_arrive_cluster(tc::map_to_rank(tc::smem_u32(&full_deq[s]), 0));
          else tc::mbar_arrive(&full_deq[s]);
        }
        if (++s == LA::kRawSt) { s = 0; ph ^= 1; }
      }
    }
  } else if (!kAnyK && warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps) {
    // ---------------------------------------------------------- dequant --
    // One thread per weight row of the CTA's tile; pair tiles (128 rows per
    // CTA): two threads per row, each decoding half of the row's K step.
    const int tid = threadIdx.x - kDeqWarp0 * 32;   // 0..255
    const int row = tid % L::kWRows;                // weight row in the CTA's part of the tile
    const int part = tid / L::kWRows;               // pair tiles: which half of the K step
    constexpr int kParts = kDeqWarps * 32 / L::kWRows;
    int s = 0, d = 0;
    uint32_t ph = 0, dph = 0;
    bool ok = true;
    for (int t = t_first; t < total_tiles && ok; t += t_step) {
      const Tile tl = get_tile<kGrouped>(p, t);
      if (!tl.valid || tl.expert < 0) continue;
      for (int kb = kb0; kb < nkb; ++kb) {
        if (!tc::mbar_wait(&full_raw[s], ph, abort_flag, p.status, kStatusTimeoutDequant) ||
            !tc::mbar_wait<kPair>(&empty_deq[d], dph ^ 1, abort_flag, p.status, kStatusTimeoutDequant)) {
          ok = false;
          break;
        }
        const uint32_t w_addr = smem_base + L::kWOff + s * L::kWBytes;
        const uint32_t b_addr = smem_base + L::kDeqOff + d * L::kDeqStride;
        if constexpr (F == Fmt::kInt8) {
          // Rows of 64 int8 codes (TMA 64-byte swizzle: chunk c at
          // c ^ ((row >> 1) & 3)) -> binary16, exactly: weight row `row`
          // (pair tiles: half of its chunks), and half of the chunks of A
          // row tid & 127 (chunks 2 (tid >> 7) and 2 (tid >> 7) + 1).
          const uint32_t a_raw = smem_base + L::kAOff + s * L::kAStride;
          const uint32_t a_dq = b_addr + L::kDeqAOff;
          const int ar = tid & (UMMA_M - 1);
          const int apart = tid >> 7;
#pragma unroll
          for (int i = 0; i < 4 / kParts; ++i) {
            const int c = part * (4 / kParts) + i;
            const uint32_t src = row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
            uint4 lo, hi;
            s8x16_to_f16(tc::lds128(w_addr + src), lo, hi);
            tc::sts128(b_addr + sw128_off(row, 2 * c), lo);
            tc::sts128(b_addr + sw128_off(row, 2 * c + 1), hi);
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 2 * apart + i;
            uint4 lo, hi;
            const uint32_t asrc = ar * 64 + ((c ^ ((ar >> 1) & 3)) << 4);
            s8x16_to_f16(tc::lds128(a_raw + asrc), lo, hi);
            tc::sts128(a_dq + sw128_off(ar, 2 * c), lo);
            tc::sts128(a_dq + sw128_off(ar, 2 * c + 1), hi);
          }
        } else if constexpr (F == Fmt::kFp8) {
          // Row of 64 codes, TMA 64-byte swizzle: chunk c sits at c ^ ((row >> 1) & 3).
#pragma unroll
          for (int i = 0; i < 4 / kParts; ++i) {
            const int c = part * (4 / kParts) + i;
            const uint4 v = tc::lds128(w_addr + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
            uint4 lo, hi;
            fp8x16_to_bf16(v, lo, hi);
            tc::sts128(b_addr + sw128_off(row, 2 * c), lo);
            tc::sts128(b_addr + sw128_off(row, 2 * c + 1), hi);
          }
        } else {
          // Row of 32 packed bytes, TMA 32-byte swizzle: chunk c at c ^ ((row >> 2) & 1).
          const uint32_t sc = tc::lds32(smem_base + L::kSOff + s * L::kScaleBytes + row * 4);
#pragma unroll
          for (int i = 0; i < 2 / kParts; ++i) {
            const int c = part * (2 / kParts) + i;
            const uint4 v = tc::lds128(w_addr + row * 32 + ((c ^ ((row >> 2) & 1)) << 4));
            const uint16_t s0 = e4m3_to_f16(sc >> (16 * c));
            const uint16_t s1 = e4m3_to_f16(sc >> (16 * c + 8));
            uint4 lo, hi;
            nvfp4x16_to_bf16(v.x, v.y, s0, lo, hi);
            tc::sts128(b_addr + sw128_off(row, 4 * c), lo);
            tc::sts128(b_addr + sw128_off(row, 4 * c + 1), hi);
            nvfp4x16_to_bf16(v.z, v.w, s1, lo, hi);
            tc::sts128(b_addr + sw128_off(row, 4 * c + 2), lo);
            tc::sts128(b_addr + sw128_off(row, 4 * c + 3), hi);
          }
        }
        tc::fence_proxy_async_smem();   // make the generic stores visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          // Pair tiles: the MMA issuer (rank 0) waits for both CTAs' rows.
          if constexpr (kPair) tc::mbar_arrive_cluster(tc::map_to_rank(tc::smem_u32(&full_deq[d]), 0));
          else tc::mbar_arrive(&full_deq[d]);
          tc::mbar_arrive(&empty_raw[s]);
        }
        if (++s == L::kRawSt) { s = 0; ph ^= 1; }
        if (++d == L::kDeqSt) { d = 0; dph ^= 1; }
      }
    }
  } else if (warp >= kEpiWarp0) {
    // --------------------------------------------------------- epilogue --
    const int g = warp & 3;                 // TMEM lane group of this warp
    int hand = 0;                           // accumulator hand-overs received
    const uint32_t stage = smem_base + L::kStageOff + g * 4096;   // this warp's 2 staging boxes
    int sbuf = 0;
    for (int t = t_first; t < total_tiles; t += t_step) {
      const Tile tl = get_tile<kGrouped>(p, t);
      if (!tl.valid) continue;
      if (tl.expert < 0) {
        // Inactive group: write zeros for its rows (all-zero bits in every
        // output type; no epilogue), no tensor-core work.
        const int es = p.ep.out_kind == kOutF32 ? 4 : 2;   // bytes per output element
        const bool vec0 = (static_cast<int64_t>(p.N) * es) % 16 == 0;
        const int per16 = 16 / es;                        // elements per 16-byte store
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int m = tl.m0 + h * kHalfRows + a_row0 + g * 32 + lane;
          if (m >= tl.m_end) continue;
          const int cend = min(BN, p.N - tl.n0);
          const int64_t o = static_cast<int64_t>(m) * p.N + tl.n0;
          int c = 0;
          if (vec0) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + o * es);
            for (; c + per16 <= cend; c += per16) dst[c / per16] = make_uint4(0u, 0u, 0u, 0u);
          }
          for (; c < cend; ++c) epi_store(p.out, o + c, p.ep.out_kind, 0.f);
        }
        continue;
      }
      // W8A8: every chunk, the tile's last included, is added to the running
      // int32 sums in the second accumulator (lane 32 g + lane, columns
      // BN + c) and the first accumulator is handed back to the MMAs; the
      // output is then formed from the int32 sums while the MMAs run the
      // next tile.
      if constexpr (F == Fmt::kInt8) {
        const int nch = (nkb - kb0 + kInt8ChunkSteps - 1) / kInt8ChunkSteps;
        const uint32_t lrow = tmem_base + (static_cast<uint32_t>(g * 32) << 16);
        bool fail = false;
        bool have_run = false;
#pragma unroll 1
        for (int j = 0; j < nch; ++j) {
          if (!tc::mbar_wait<kPair>(&tmem_full[0], hand & 1, abort_flag, p.status, kStatusTimeoutEpilogue)) {
            fail = true;
            break;
          }
          ++hand;
          tc::tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t r[32], y[32];
            tc::tmem_ld_32x32b_x32(lrow + c0, r);
            if (have_run) tc::tmem_ld_32x32b_x32(lrow + BN + c0, y);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = static_cast<uint32_t>(chunk_sum(r[i], have_run ? y[i] : 0u, have_run));
            tc::tmem_st_32x32b_x32(lrow + BN + c0, y);
          }
          tc::tmem_wait_st();
          have_run = true;
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair) tc::mbar_arrive_cluster(tc::map_to_rank(tc::smem_u32(&tmem_empty[0]), 0));
            else tc::mbar_arrive(&tmem_empty[0]);
          }
        }
        if (fail) break;
      } else {
        if (!tc::mbar_wait<kPair>(&tmem_full[0], hand & 1, abort_flag, p.status, kStatusTimeoutEpilogue)) break;
        ++hand;
        tc::tc_fence_after();
      }
      if (split) {
        // This CTA's raw fp32 partial of rows [0, 128) -> shared memory (the
        // operand rings are idle now: every MMA has completed).  Rows are
        // padded to kPartStride bytes so that 8 consecutive rows hit
        // distinct banks.  The cluster reduction at the end of the kernel sums
        // the partials of all ranks.
        // W8A8: the partial is the exact int32 sum in the second
        // accumulator (bits stored; the reduction adds int32).
        const int r_local = g * 32 + lane;
        const uint32_t prow = smem_base + r_local * kPartStride;
        constexpr uint32_t kAccCol = F == Fmt::kInt8 ? BN : 0;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(g * 32) << 16) + kAccCol + c0, r);
          tc::tmem_wait_ld();
          if (tl.m0 + r_local < tl.m_end) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              tc::sts128(prow + (c0 + 4 * i) * 4, make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]));
          }
        }
        if constexpr (F != Fmt::kInt8) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tmem_empty[0]);
        }
        continue;
      }
      const bool plain_epi = epi_plain(p.ep);
      const bool vec_ok = p.ep.out_kind == kOutF32 ? (p.N % 4 == 0) : (p.N % 8 == 0);
      const int64_t bias0 = static_cast<int64_t>(tl.expert) * p.ep.bias_stride;   // bias row of the expert
      const bool residue_rows = kAnyK && !p.a_tma;
      // W8A8: one half of output rows, from the int32 sums in the second accumulator.
      const int halves = F == Fmt::kInt8 ? 1 : (residue_rows || tl.m_end - tl.m0 > kHalfRows) ? 2 : 1;
#pragma unroll 1
      for (int h = 0; h < halves; ++h) {
        // Lane 32 g + lane of TMEM half h holds tile row h * 128 + 32 g + lane
        // (pair tiles: h * 256 + 128 rank + 32 g + lane), or (any K, residue
        // order) tile row 8 lane + 4 h + g.
        const int srow = 128 * h + 32 * g + lane;   // residue order: class srow / rr, group srow % rr
        const int rlog = 8 - (__ffs(p.a_res) - 1);
        const int m = residue_rows ? tl.m0 + a_row0 + p.a_res * (srow & ((1 << rlog) - 1)) + (srow >> rlog)
                                   : tl.m0 + h * kHalfRows + a_row0 + g * 32 + lane;
        const bool row_ok = m < tl.m_end;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(g * 32) << 16) + h * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(taddr + (F == Fmt::kInt8 ? BN : 0) + c0, r);
          tc::tmem_wait_ld();
          const int n = tl.n0 + c0;
          float v[32];
          if constexpr (F == Fmt::kInt8) {
            // acc = the exact int32 sum, then (float(acc) * a_scale[m]) *
            // b_scale[n], each step rounded once; lane i loads b_scale of
            // column n + i and the warp shares it (every lane of the warp is
            // here: the row test comes after).
            const float sbv = n + lane < p.N ? __ldg(p.b_scale + n + lane) : 0.f;
            const float sa = row_ok ? __ldg(p.a_scale + m) : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = __fmul_rn(__fmul_rn(__int2float_rn(static_cast<int>(r[i])), sa),
                               __shfl_sync(0xFFFFFFFFu, sbv, i));
          }
          // TMA store of the warp's 32 x 32 box (16-bit outputs, all rows of
          // the box inside the tile or, for the plain GEMM, past the end of
          // the output where the store clips them): every lane stages its row.
          const int mbox = tl.m0 + h * kHalfRows + a_row0 + g * 32;
          const bool use_box = L::kStageBytes > 0 && !kAnyK && p.tma_out && n < p.N &&
                               mbox < tl.m_end && (!kGrouped || mbox + 32 <= tl.m_end);
          if (use_box) {
            const int lim = min(32, p.N - n);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = tl.scale * __uint_as_float(r[i]);
            if (!plain_epi) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = epi_apply(p.ep, v[i], bias0 + n + (i < lim ? i : 0));
            }
            const uint32_t buf = stage + sbuf * 2048;
            if (lane == 0) tc::bulk_wait_read<1>();   // the store from this buffer two boxes ago has read it
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w4[4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                w4[q] = p.ep.out_kind == kOutBf16 ? pack_bf16x2(v[8 * j + 2 * q], v[8 * j + 2 * q + 1])
                                                  : pack_f16x2(v[8 * j + 2 * q], v[8 * j + 2 * q + 1]);
              tc::sts128(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4),
                         make_uint4(w4[0], w4[1], w4[2], w4[3]));
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tc::tma_store_2d(&tmap_o, buf, n, mbox);
              tc::bulk_commit();
            }
            sbuf ^= 1;
            continue;
          }
          if (!row_ok || n >= p.N) continue;
          const int lim = min(32, p.N - n);
          if constexpr (F != Fmt::kInt8) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = tl.scale * __uint_as_float(r[i]);
          }
          if (!plain_epi) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = epi_apply(p.ep, v[i], bias0 + n + (i < lim ? i : 0));
          }
          const int64_t o = static_cast<int64_t>(m) * p.N + n;
          if (vec_ok && lim == 32) {
            if (p.ep.out_kind == kOutF32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            } else if (p.ep.out_kind == kOutBf16) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + o);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                    pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + o);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack_f16x2(v[8 * i], v[8 * i + 1]), pack_f16x2(v[8 * i + 2], v[8 * i + 3]),
                                    pack_f16x2(v[8 * i + 4], v[8 * i + 5]), pack_f16x2(v[8 * i + 6], v[8 * i + 7]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < lim) epi_store(p.out, o + i, p.ep.out_kind, v[i]);
          }
        }
      }
      if constexpr (F != Fmt::kInt8) {   // (W8A8 handed the accumulator back after its last chunk)
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) tc::mbar_arrive_cluster(tc::map_to_rank(tc::smem_u32(&tmem_empty[0]), 0));
          else tc::mbar_arrive(&tmem_empty[0]);
        }
      }
    }
    // Every TMA store of this warp has completed before the CTA exits.
    if (lane == 0) tc::bulk_wait_all();
    __syncwarp();
  }

  tc::tc_fence_before();
  __syncthreads();
  if (split) {
    // Split-K reduction across the cluster through distributed shared
    // memory: rank r sums columns [r * BN / S, (r + 1) * BN / S) of the tile
    // over all ranks in rank order (deterministic), scales, converts, stores.
    tc::cluster_sync();
    if (t_first < total_tiles && !*abort_flag) {   // an aborted CTA has no partial
      const Tile tl = get_tile<kGrouped>(p, t_first);
      const int rows = tl.m_end - tl.m0;
      const int cols = BN / p.ksplit;                 // multiple of 4 (host check)
      const int c_begin = crank * cols;
      const int groups = rows * (cols / 4);
      for (int task = threadIdx.x; task < groups; task += kThreads) {
        const int r = task / (cols / 4);
        const int c = c_begin + 4 * (task % (cols / 4));
        const uint32_t local = smem_base + r * kPartStride + c * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int iacc[4] = {0, 0, 0, 0};   // W8A8: exact int32 sums of the ranks' partials
        // every rank's partial requested before the first add (the loads are
        // in flight together), then summed in rank order
        float4 part[kMaxClusterSplit];
#pragma unroll
        for (int q = 0; q < kMaxClusterSplit; ++q)
          if (q < p.ksplit) part[q] = tc::ld_cluster_f4(tc::map_to_rank(local, q));
#pragma unroll
        for (int q = 0; q < kMaxClusterSplit; ++q) {
          if (q >= p.ksplit) break;
          const float4 v = part[q];
          if constexpr (F == Fmt::kInt8) {
            iacc[0] += __float_as_int(v.x); iacc[1] += __float_as_int(v.y);
            iacc[2] += __float_as_int(v.z); iacc[3] += __float_as_int(v.w);
          } else {
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
        }
        const int m = tl.m0 + r;
        const int n = tl.n0 + c;
        float o[4] = {p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w};
        if constexpr (F == Fmt::kInt8) {
          const float sa = __ldg(p.a_scale + m);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o[i] = __fmul_rn(__fmul_rn(__int2float_rn(iacc[i]), sa),
                             __ldg(p.b_scale + min(n + i, p.N - 1)));
        }
        const int64_t base = static_cast<int64_t>(m) * p.N + n;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n + i < p.N) epi_store(p.out, base + i, p.ep.out_kind, epi_apply(p.ep, o[i], n + i));
      }
    }
    tc::cluster_sync();   // no CTA leaves while a peer still reads its partial
  }
  // Pair tiles: neither CTA frees its TMEM or leaves while rank 0's MMAs may
  // still read the peer's shared memory or a remote arrival is on its way.
  if constexpr (kPair) tc::cluster_sync();
  if (warp == kWarpMma) {
    tc::tc_fence_after();
    if constexpr (kPair) tc::tmem_dealloc_pair(tmem_base, kTmemCols);
    else tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// K = 0 (the sum is empty): out[m, n] = epilogue(alpha * 0) for the column n.
__global__ void k_fill_scaled_zero(void* out, Epi ep, int64_t count, int64_t N, float alpha) {
  const float v = alpha * 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    epi_store(out, i, ep.out_kind, epi_apply(ep, v, i % N));
}

// --------------------------------------------------------------- host --

template <Fmt F, bool kGrouped, bool kAnyK = false, bool kPair = false>
cudaError_t launch(const Ctx& c, const CUtensorMap& ta, const CUtensorMap& tw, const uint8_t* scales,
                   const Problem& p, int grid, const CUtensorMap* tx = nullptr,
                   const CUtensorMap* to = nullptr) {
  auto kern = k_wq_gemm<F, kGrouped, kAnyK, kPair>;
  const uint32_t smem = SmemFor<F, kAnyK, kPair>::kAlloc;
  Problem pl = p;
  pl.stall_producer = c.test_stall_producer ? 1 : 0;
  // The shared-memory opt-in is set once per device (it is not a stream
  // operation, so it is kept out of any CUDA-graph capture after the first call).
  static std::atomic<uint64_t> configured{0};
  const uint64_t bit = 1ull << (c.device & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : p.ksplit > 1 ? p.ksplit : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (kPair || p.ksplit > 1) ? 1 : 0;
  CUtensorMap unused;
  memset(&unused, 0, sizeof(unused));
  return cudaLaunchKernelEx(&cfg, kern, ta, tw, tx ? *tx : unused, to ? *to : unused, scales, pl);
}

// CTA pairs (clusters of 2 one-CTA-per-SM blocks) the GPU holds at once,
// queried once per device (pair kernels of both formats have one CTA per SM).
int max_pairs(const Ctx& c) {
  static std::atomic<int> cached[64];
  const int dev = c.device & 63;
  int v = cached[dev].load(std::memory_order_acquire);
  if (v > 0) return v;
  auto kern = k_wq_gemm<Fmt::kFp8, false, false, true>;
  const uint32_t smem = SmemPair<Fmt::kFp8>::kAlloc;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (c.num_sms / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  v = n > 0 ? std::min(n, c.num_sms / 2) : std::max(1, c.num_sms / 2);
  cached[dev].store(v, std::memory_order_release);
  return v;
}

cudaError_t fill_zero(const Ctx& c, void* out, const Epi& ep, int64_t count, int64_t N, float alpha) {
  const int grid = static_cast<int>(std::min<int64_t>((count + 255) / 256, c.num_sms * 8LL));
  k_fill_scaled_zero<<<grid > 0 ? grid : 1, 256, 0, c.stream>>>(out, ep, count, N > 0 ? N : 1, alpha);
  return cudaGetLastError();
}

// The output tensor map for TMA stores of the epilogue's 32 x 32 boxes:
// 16-bit outputs whose rows are 16-byte strided (N % 8 == 0).  Returns
// whether it was made (1) or the epilogue stores directly (0).
int output_map(const Epi& ep, void* out, int64_t rows, int64_t N, CUtensorMap* to) {
  memset(to, 0, sizeof(*to));
  if (ep.out_kind == kOutF32 || N % 8 != 0 || rows <= 0 || N <= 0) return 0;
  const auto dt = ep.out_kind == kOutBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return encode_2d(to, dt, out, N, rows, N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ? 1 : 0;
}

Problem base_problem(const Ctx& c, void* out, const Epi& ep, int64_t M, int64_t N, int64_t K,
                     float alpha) {
  Problem p{};
  p.out = out;
  p.status = c.status;
  p.alpha = alpha;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.bm = BM;
  p.num_n_tiles = static_cast<int>((N + BN - 1) / BN);
  p.num_k_blocks = static_cast<int>((K + BK - 1) / BK);
  p.ep = ep;
  p.ksplit = 1;
  p.kb_per_split = p.num_k_blocks;
  return p;
}

// Small M: too few tiles to fill the GPU.  Split K over a cluster of up to 4
// CTAs (clusters of 8 one-CTA-per-SM blocks do not all fit in one wave) when each tile has at most 128 rows (one MMA half; the partials fit in
// shared memory) and every split gets at least 4 K steps.  Returns the grid.
int plan_split(const Ctx& c, Problem& p, int tiles) {
  if (p.M > UMMA_M || tiles * 2 > c.num_sms) return std::min(tiles, c.num_sms);
  int s = std::min(4, c.num_sms / tiles);
  s = std::min(s, p.num_k_blocks / 4);
  while (s > 1 && (BN / s) % 4 != 0) --s;
  if (s < 2) return std::min(tiles, c.num_sms);
  const int per = (p.num_k_blocks + s - 1) / s;
  s = (p.num_k_blocks + per - 1) / per;           // no empty split
  if (s < 2 || (BN / s) % 4 != 0) return std::min(tiles, c.num_sms);
  p.ksplit = s;
  p.kb_per_split = per;
  return tiles * s;
}

}  // namespace

cudaError_t launch_fp8_gemm(const Ctx& c, void* out, const Epi& ep, const void* a, const uint8_t* w,
                            int64_t M, int64_t N, int64_t K, float alpha) {
  if (K == 0) return fill_zero(c, out, ep, M * N, N, alpha);
  if (K % 16 != 0) {
    // Rows not 16-byte strided: rows 8 (A) and 16 (W) apart are.  Tensor maps
    // over the full groups (any M, no split-K).
    CUtensorMap ta, tx, tw;
    memset(&ta, 0, sizeof(ta));
    memset(&tx, 0, sizeof(tx));
    memset(&tw, 0, sizeof(tw));
    Problem p = base_problem(c, out, ep, M, N, K, alpha);
    p.a_g = a;
    p.w_g = w;
    p.a_tma = K % 8 == 0 ? 1 : 0;
    // A rows a_res apart are 16-byte strided (2 a_res K % 16 == 0).
    p.a_res = (K & 1) ? 8 : (K & 3) ? 4 : 2;
    p.a_groups = p.a_tma ? 0 : static_cast<int>(M / p.a_res);
    // W rows w_res apart are 16-byte strided (w_res * K % 16 == 0).
    p.w_res = (K & 1) ? 16 : (K & 3) ? 8 : (K & 7) ? 4 : 2;
    p.w_groups = static_cast<int>(N / p.w_res);
    if (p.a_tma && !encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, M, K * 2, BK, BM,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (p.a_groups > 0 &&
        (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, p.a_res * K, M / p.a_res, 2 * p.a_res * K,
                    72, any_a_in_place(p.a_res), CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, p.a_res * K, M / p.a_res, 2 * p.a_res * K,
                    72, 256 / p.a_res - any_a_in_place(p.a_res), CU_TENSOR_MAP_SWIZZLE_NONE)))
      return cudaErrorInvalidValue;
    // M > 256: pair tiles (each CTA realigns its 256 rows of A and decodes
    // 128 weight rows: W boxes of 8 groups).
    const bool pair = M > BM;
    if (p.w_groups > 0 &&
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, p.w_res * K, N / p.w_res, p.w_res * K,
                   kAnyRowW, (pair ? kPairWRows : BN) / p.w_res, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    if (pair) {
      p.bm = kPairBM;
      const int tiles = ((p.M + kPairBM - 1) / kPairBM) * p.num_n_tiles;
      return launch<Fmt::kFp8, false, true, true>(c, ta, tw, nullptr, p,
                                                   2 * std::min(tiles, max_pairs(c)), &tx);
    }
    const int tiles = ((p.M + BM - 1) / BM) * p.num_n_tiles;
    return launch<Fmt::kFp8, false, true>(c, ta, tw, nullptr, p, std::min(tiles, c.num_sms), &tx);
  }
  if (fewrow_ok(0, M, K, a, w, nullptr)) return launch_fp8_gemm_fewrow(c, out, ep, a, w, M, N, K, alpha);
  if (M <= skinny_max_rows()) return launch_fp8_gemm_skinny(c, out, ep, a, w, M, N, K, alpha);
  // Pair tiles: A in 128-row boxes, each CTA's 128 weight rows in one box.
  CUtensorMap ta, tw;
  if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, M, K * 2, BK, UMMA_M,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K, N, K, BK, kPairWRows,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  Problem p = base_problem(c, out, ep, M, N, K, alpha);
  p.bm = kPairBM;
  const int tiles = ((p.M + kPairBM - 1) / kPairBM) * p.num_n_tiles;
  const int grid = 2 * std::min(tiles, max_pairs(c));
  CUtensorMap to;
  p.tma_out = output_map(ep, out, M, N, &to);
  return launch<Fmt::kFp8, false, false, true>(c, ta, tw, nullptr, p, grid, nullptr, &to);
}

cudaError_t launch_nvfp4_gemm(const Ctx& c, void* out, const Epi& ep, const void* a,
                              const uint8_t* q, const uint8_t* bs, int64_t M, int64_t N, int64_t K,
                              float alpha) {
  if (K == 0) return fill_zero(c, out, ep, M * N, N, alpha);
  if (fewrow_ok(1, M, K, a, q, bs))
    return launch_nvfp4_gemm_fewrow(c, out, ep, a, q, bs, M, N, K, alpha);
  if (M <= skinny_max_rows() && nvfp4_skinny_ok(bs, K))
    return launch_nvfp4_gemm_skinny(c, out, ep, a, q, bs, M, N, K, alpha);
  if (M > UMMA_M) {
    // Pair tiles, as launch_fp8_gemm.
    CUtensorMap ta, tw;
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, M, K * 2, BK, UMMA_M,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K / 2, N, K / 2, BK / 2, kPairWRows,
                   CU_TENSOR_MAP_SWIZZLE_32B))
      return cudaErrorInvalidValue;
    Problem p = base_problem(c, out, ep, M, N, K, alpha);
    p.bm = kPairBM;
    const int tiles = ((p.M + kPairBM - 1) / kPairBM) * p.num_n_tiles;
    const int grid = 2 * std::min(tiles, max_pairs(c));
    CUtensorMap to;
    p.tma_out = output_map(ep, out, M, N, &to);
    return launch<Fmt::kNvfp4, false, false, true>(c, ta, tw, bs, p, grid, nullptr, &to);
  }
  CUtensorMap ta, tw;
  if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, M, K * 2, BK, BM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K / 2, N, K / 2, BK / 2, BN,
                 CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  Problem p = base_problem(c, out, ep, M, N, K, alpha);
  const int tiles = ((p.M + BM - 1) / BM) * p.num_n_tiles;
  const int grid = plan_split(c, p, tiles);
  CUtensorMap to;
  p.tma_out = output_map(ep, out, M, N, &to);
  return launch<Fmt::kNvfp4, false>(c, ta, tw, bs, p, grid, nullptr, &to);
}

cudaError_t launch_int8_gemm(const Ctx& c, void* out, const Epi& ep, const int8_t* a,
                             const int8_t* b, const float* a_scale, const float* b_scale,
                             int64_t M, int64_t N, int64_t K) {
  // K = 0: every sum is 0, so the output is the epilogue of 0.
  if (K == 0) return fill_zero(c, out, ep, M * N, N, 0.f);
  if (K > kInt8MaxK) return cudaErrorInvalidValue;   // refused earlier by the C ABI
  if (M > UMMA_M) {
    // Pair tiles: 256 output rows (128 A rows per CTA) x 256 weight rows.
    CUtensorMap ta, tw;
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, BK, UMMA_M, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, BK, kPairWRows,
                   CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    Problem p = base_problem(c, out, ep, M, N, K, 1.0f);
    p.bm = 2 * UMMA_M;
    p.a_scale = a_scale;
    p.b_scale = b_scale;
    const int tiles = ((p.M + p.bm - 1) / p.bm) * p.num_n_tiles;
    return launch<Fmt::kInt8, false, false, true>(c, ta, tw, nullptr, p, 2 * std::min(tiles, max_pairs(c)));
  }
  CUtensorMap ta, tw;
  if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, BK, UMMA_M, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, BK, BN, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  Problem p = base_problem(c, out, ep, M, N, K, 1.0f);
  p.bm = UMMA_M;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  const int tiles = ((p.M + UMMA_M - 1) / UMMA_M) * p.num_n_tiles;
  const int grid = plan_split(c, p, tiles);
  return launch<Fmt::kInt8, false>(c, ta, tw, nullptr, p, grid);
}

// The grouped problem shared by both formats, and its persistent grid: an
// upper bound of the work list (the exact count needs the device offsets),
// capped at one CTA per SM.  (Pair tiles of 512 rows were measured slower
// here: experts of 500-570 rows leave 30-60-row tails that cost a 256-row
// pair MMA half each, 1.34x padded MMA rows against 1.14x with 256-row
// one-CTA tiles.)
static Problem grouped_problem(const Ctx& c, void* out, const Epi& ep, const uint32_t* a_offsets,
                               const int32_t* expert_ids, const float* expert_scales, int64_t G,
                               int64_t E, int64_t max_rows, int64_t total_M, int64_t N, int64_t K,
                               int* grid) {
  Problem p = base_problem(c, out, ep, total_M, N, K, 1.0f);
  p.a_offsets = a_offsets;
  p.expert_ids = expert_ids;
  p.expert_scales = expert_scales;
  p.G = static_cast<int>(G);
  p.E = (K > 0) ? static_cast<int>(E) : 0;
  p.max_rows = static_cast<int>(std::min<int64_t>(max_rows, total_M));
  const int64_t mt = (p.max_rows + BM - 1) / BM;
  const int64_t bound = std::min<int64_t>(G * mt * p.num_n_tiles, 1LL << 30);
  *grid = std::max(1, static_cast<int>(std::min<int64_t>(bound, c.num_sms)));
  return p;
}

cudaError_t launch_fp8_grouped_gemm(const Ctx& c, void* out, const Epi& ep, const void* a,
                                    const uint8_t* w, const uint32_t* a_offsets,
                                    const int32_t* expert_ids, const float* expert_scales,
                                    int64_t G, int64_t E, int64_t max_rows, int64_t total_M,
                                    int64_t N, int64_t K) {
  // With no weights or an empty sum every covered row is zero: the kernel's
  // zero path handles that when no expert is valid (E = 0), and no tensor map
  // is touched.
  CUtensorMap ta, tw;
  memset(&ta, 0, sizeof(ta));
  memset(&tw, 0, sizeof(tw));
  if (E > 0 && K > 0) {
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, total_M, K * 2, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&tw, w, K, N, E, BK, BN, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  int grid = 1;
  Problem p = grouped_problem(c, out, ep, a_offsets, expert_ids, expert_scales, G, E,
                              max_rows, total_M, N, K, &grid);
  CUtensorMap to;
  p.tma_out = output_map(ep, out, total_M, N, &to);
  return launch<Fmt::kFp8, true>(c, ta, tw, nullptr, p, grid, nullptr, &to);
}

cudaError_t launch_nvfp4_grouped_gemm(const Ctx& c, void* out, const Epi& ep, const void* a,
                                      const uint8_t* q, const uint8_t* bs, const uint32_t* a_offsets,
                                      const int32_t* expert_ids, const float* expert_scales,
                                      int64_t G, int64_t E, int64_t max_rows, int64_t total_M,
                                      int64_t N, int64_t K) {
  // As launch_fp8_grouped_gemm, with the packed expert stack q [E, N, K/2]
  // (3-D tensor map, 32-byte swizzle) and block scales bs [E, N, K/16].
  CUtensorMap ta, tw;
  memset(&ta, 0, sizeof(ta));
  memset(&tw, 0, sizeof(tw));
  if (E > 0 && K > 0) {
    if (!encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, total_M, K * 2, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&tw, q, K / 2, N, E, BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_32B))
      return cudaErrorInvalidValue;
  }
  int grid = 1;
  Problem p = grouped_problem(c, out, ep, a_offsets, expert_ids, expert_scales, G, E,
                              max_rows, total_M, N, K, &grid);
  CUtensorMap to;
  p.tma_out = output_map(ep, out, total_M, N, &to);
  return launch<Fmt::kNvfp4, true>(c, ta, tw, bs, p, grid, nullptr, &to);
}

}  // namespace gq
