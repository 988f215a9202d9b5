// internal.h -- host-side declarations shared between the gq translation units.
// Not part of the public C ABI (that is include/gq.h).
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace gq {

// Output type and fused epilogue of a product kernel:
//   out = act(alpha * acc + bias[n]) converted to out_kind (round to nearest even).
enum : int { kOutF32 = 0, kOutBf16 = 1, kOutF16 = 2 };
enum : int { kActNone = 0, kActRelu = 1, kActSilu = 2, kActGeluTanh = 3 };

struct Epi {
  const void* bias;      // [N] (grouped: [E, N], row e for expert e), or nullptr
  int64_t bias_stride;   // elements between experts' bias rows (grouped), else 0
  int bias_kind;         // element type of bias: kOutF32 / kOutBf16 / kOutF16
  int act;               // kAct*
  int out_kind;          // kOut*
};

// Per-call launch context filled by the C-ABI layer.
struct Ctx {
  cudaStream_t stream;
  uint32_t* status;   // device address of the per-device status word (then the wait limit)
  int num_sms;        // multiprocessor count of the current device
  int device;
  bool overlap_weights;  // GQ_LAUNCH_OVERLAP_WEIGHT_READS is set (gq_set_launch_flags)
  bool test_stall_producer;  // GQ_LAUNCH_TEST_STALL_PRODUCER is set (tests only)
};

// Launch `kern` on c.stream.  With `pdl` the launch carries the programmatic
// stream serialization attribute: the kernel may start before the previous
// kernel in the stream finishes and must call pdl_wait() before touching
// memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const Ctx& c, bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block,
                          size_t smem, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// materialize.cu
cudaError_t launch_fp8_materialize(const Ctx& c, void* out, int out_kind,
                                   const uint8_t* w, int64_t total);
cudaError_t launch_nvfp4_materialize(const Ctx& c, void* out, int out_kind,
                                     const uint8_t* q, const uint8_t* bs,
                                     int64_t total_blocks);

// gemv.cu
cudaError_t launch_fp8_gemv(const Ctx& c, void* y, const Epi& ep, const void* x,
                            const uint8_t* w, int64_t N, int64_t K, float alpha);
cudaError_t launch_nvfp4_gemv(const Ctx& c, void* y, const Epi& ep, const void* x,
                              const uint8_t* q, const uint8_t* bs, int64_t N,
                              int64_t K, float alpha);

// The GEMVs' launch shapes with only the weight (and block-scale) loads:
// format 0 = FP8 (K % 16 == 0), 1 = NVFP4.  Writes a checksum per row to y (bf16).
cudaError_t launch_gemv_read_floor(const Ctx& c, int format, void* y, const uint8_t* w,
                                   const uint8_t* bs, int64_t N, int64_t K);

// gemm.cu
cudaError_t launch_fp8_gemm(const Ctx& c, void* out, const Epi& ep, const void* a,
                            const uint8_t* w, int64_t M, int64_t N, int64_t K,
                            float alpha);
cudaError_t launch_nvfp4_gemm(const Ctx& c, void* out, const Epi& ep, const void* a,
                              const uint8_t* q, const uint8_t* bs, int64_t M,
                              int64_t N, int64_t K, float alpha);
cudaError_t launch_fp8_grouped_gemm(const Ctx& c, void* out, const Epi& ep,
                                    const void* a, const uint8_t* w,
                                    const uint32_t* a_offsets,
                                    const int32_t* expert_ids,
                                    const float* expert_scales, int64_t G,
                                    int64_t E, int64_t max_rows,
                                    int64_t total_M, int64_t N, int64_t K);

// W8A8: c = epilogue((acc * a_scale[m]) * b_scale[n]), acc = sum a[m,k] b[n,k]
// exactly in int32, for K <= kInt8MaxK (128 * 128 * kInt8MaxK < 2^31).
constexpr int64_t kInt8MaxK = 130560;
cudaError_t launch_int8_gemm(const Ctx& c, void* out, const Epi& ep, const int8_t* a,
                             const int8_t* b, const float* a_scale, const float* b_scale,
                             int64_t M, int64_t N, int64_t K);
// Per-row absmax int8 quantization of bf16 activations.
cudaError_t launch_int8_quantize_rows(const Ctx& c, int8_t* q, float* scale, const void* x,
                                      int64_t M, int64_t K);
cudaError_t launch_nvfp4_grouped_gemm(const Ctx& c, void* out, const Epi& ep,
                                      const void* a, const uint8_t* q,
                                      const uint8_t* bs, const uint32_t* a_offsets,
                                      const int32_t* expert_ids,
                                      const float* expert_scales, int64_t G,
                                      int64_t E, int64_t max_rows,
                                      int64_t total_M, int64_t N, int64_t K);

// fewrow.cu (1 <= M <= 16): register-fed mma.sync products.  fewrow_ok says
// whether the kernel takes the call (format 0 = FP8: K % 64 == 0; 1 = NVFP4:
// K % 128 == 0; a and w 16-byte aligned, NVFP4 bs 2-byte aligned).
bool fewrow_ok(int format, int64_t M, int64_t K, const void* a, const uint8_t* w,
               const uint8_t* bs);
cudaError_t launch_fp8_gemm_fewrow(const Ctx& c, void* out, const Epi& ep, const void* a,
                                   const uint8_t* w, int64_t M, int64_t N, int64_t K,
                                   float alpha);
cudaError_t launch_nvfp4_gemm_fewrow(const Ctx& c, void* out, const Epi& ep, const void* a,
                                     const uint8_t* q, const uint8_t* bs, int64_t M, int64_t N,
                                     int64_t K, float alpha);

// gemm_skinny.cu (M <= skinny_max_rows())
int skinny_max_rows();
bool nvfp4_skinny_ok(const uint8_t* bs, int64_t K);   // the NVFP4 few-row kernel takes this K
cudaError_t launch_fp8_gemm_skinny(const Ctx& c, void* out, const Epi& ep, const void* a,
                                   const uint8_t* w, int64_t M, int64_t N, int64_t K,
                                   float alpha);
cudaError_t launch_nvfp4_gemm_skinny(const Ctx& c, void* out, const Epi& ep, const void* a,
                                     const uint8_t* q, const uint8_t* bs, int64_t M,
                                     int64_t N, int64_t K, float alpha);

// api.cu: the driver's cuTensorMapEncodeTiled, resolved once at run time so
// that the library does not link against libcuda.
void* tensor_map_encode_fn();

}  // namespace gq
