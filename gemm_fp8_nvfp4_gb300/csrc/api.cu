// api.cu -- the C ABI of libgq (declared in include/gq.h).
//
// Host-side only: argument checks, the per-device context (SM count, device
// status word), and dispatch to the kernel launchers of the other
// translation units.  No allocation, no synchronization (except
// gq_device_status, which is documented as synchronizing).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/gq.h"
#include "internal.h"

namespace gq {

// Per-device record: the status word (bits of waits that ran out) and the
// wait limit in ns that the kernels' bounded waits read (0 = the default).
struct __align__(16) DeviceRecord {
  uint32_t status;
  uint32_t reserved;
  uint64_t wait_limit_ns;
};
__device__ DeviceRecord g_device_record;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 = unknown, 1 = ready (sm_103), 2 = unsupported
  int num_sms = 0;
  uint32_t* status = nullptr;
};

DeviceInfo g_devices[kMaxDevices];
std::atomic<uint32_t> g_launch_flags{0};

// Fills `ctx` for the current device; returns GQ_OK or GQ_ERR_DEVICE.
int device_ctx(cudaStream_t stream, Ctx* ctx) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GQ_ERR_DEVICE;
  }
  DeviceInfo& d = g_devices[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    void* status = nullptr;
    ok = ok && major == 10 && minor == 3;
    ok = ok && cudaGetSymbolAddress(&status, g_device_record) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      d.state.store(2, std::memory_order_release);
      return GQ_ERR_DEVICE;
    }
    d.num_sms = sms;
    d.status = static_cast<uint32_t*>(status);
    d.state.store(1, std::memory_order_release);
    st = 1;
  }
  if (st != 1) return GQ_ERR_DEVICE;
  ctx->stream = stream;
  ctx->status = d.status;
  ctx->num_sms = d.num_sms;
  ctx->device = dev;
  const uint32_t flags = g_launch_flags.load(std::memory_order_relaxed);
  ctx->overlap_weights = (flags & GQ_LAUNCH_OVERLAP_WEIGHT_READS) != 0;
  ctx->test_stall_producer = (flags & GQ_LAUNCH_TEST_STALL_PRODUCER) != 0;
  return GQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_dtype(int t) { return t == GQ_F32 || t == GQ_BF16 || t == GQ_F16; }

int out_size(int t) { return t == GQ_F32 ? 4 : 2; }

// Checks an epilogue and builds the kernels' descriptor.  bias_stride is the
// distance between experts' bias rows (grouped) or 0.
int make_epi(int out_dtype, const gq_epilogue* e, int64_t bias_stride, Epi* ep) {
  ep->bias = nullptr;
  ep->bias_stride = 0;
  ep->bias_kind = kOutF32;
  ep->act = kActNone;
  ep->out_kind = out_dtype == GQ_BF16 ? kOutBf16 : (out_dtype == GQ_F16 ? kOutF16 : kOutF32);
  if (e == nullptr) return GQ_OK;
  if (e->activation < GQ_ACT_NONE || e->activation > GQ_ACT_GELU_TANH) return GQ_ERR_EPILOGUE;
  ep->act = e->activation;
  if (e->bias != nullptr) {
    if (!valid_dtype(e->bias_dtype)) return GQ_ERR_EPILOGUE;
    if (!aligned(e->bias, static_cast<uintptr_t>(out_size(e->bias_dtype)))) return GQ_ERR_ALIGN;
    ep->bias = e->bias;
    ep->bias_stride = bias_stride;
    ep->bias_kind = e->bias_dtype == GQ_BF16 ? kOutBf16 : (e->bias_dtype == GQ_F16 ? kOutF16 : kOutF32);
  }
  return GQ_OK;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return GQ_OK;
  cudaGetLastError();
  return GQ_ERR_LAUNCH;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int> g_encode_state{0};

}  // namespace

void* tensor_map_encode_fn() {
  if (g_encode_state.load(std::memory_order_acquire) == 1) return reinterpret_cast<void*>(g_encode);
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                       cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  g_encode_state.store(1, std::memory_order_release);
  return fn;
}

}  // namespace gq

using gq::aligned;
using gq::make_epi;
using gq::out_size;
using gq::valid_dtype;

extern "C" {

const char* gq_status_str(int s) {
  switch (s) {
    case GQ_OK: return "GQ_OK";
    case GQ_ERR_NULL: return "GQ_ERR_NULL: a required pointer is NULL";
    case GQ_ERR_SHAPE: return "GQ_ERR_SHAPE: a size is negative or breaks a format rule";
    case GQ_ERR_ALIGN: return "GQ_ERR_ALIGN: a pointer is not aligned as required";
    case GQ_ERR_DTYPE: return "GQ_ERR_DTYPE: unknown output dtype";
    case GQ_ERR_DEVICE: return "GQ_ERR_DEVICE: current device is not an sm_103 GPU";
    case GQ_ERR_LAUNCH: return "GQ_ERR_LAUNCH: kernel launch failed";
    case GQ_ERR_TOO_LARGE: return "GQ_ERR_TOO_LARGE: a size exceeds what the kernel supports";
    case GQ_ERR_EPILOGUE: return "GQ_ERR_EPILOGUE: unknown activation or bias dtype";
    default: return "unknown gq status";
  }
}

const char* gq_version(void) { return "gq 0.1.0 sm_103a"; }

int gq_set_launch_flags(uint32_t flags) {
  if (flags & ~static_cast<uint32_t>(GQ_LAUNCH_OVERLAP_WEIGHT_READS | GQ_LAUNCH_TEST_STALL_PRODUCER))
    return GQ_ERR_SHAPE;
  gq::g_launch_flags.store(flags, std::memory_order_relaxed);
  return GQ_OK;
}

uint32_t gq_get_launch_flags(void) { return gq::g_launch_flags.load(std::memory_order_relaxed); }

int gq_fp8_gemv_ex(void* y, int out_dtype, const void* x, const uint8_t* w, int64_t N,
                   int64_t K, float alpha, const gq_epilogue* epilogue, cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (N < 0 || K < 0) return GQ_ERR_SHAPE;
  if (N == 0) return GQ_OK;
  if (!y || (K > 0 && (!x || !w))) return GQ_ERR_NULL;
  if (!aligned(x, 2) || !aligned(y, out_size(out_dtype))) return GQ_ERR_ALIGN;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, 0, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_fp8_gemv(c, y, ep, x, w, N, K, alpha));
}

int gq_fp8_gemv(void* y, int out_dtype, const void* x, const uint8_t* w, int64_t N, int64_t K,
                float alpha, cudaStream_t stream) {
  return gq_fp8_gemv_ex(y, out_dtype, x, w, N, K, alpha, nullptr, stream);
}

int gq_nvfp4_gemv_ex(void* y, int out_dtype, const void* x, const uint8_t* q, const uint8_t* bs,
                     int64_t N, int64_t K, float alpha, const gq_epilogue* epilogue,
                     cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (N < 0 || K < 0 || K % 16 != 0) return GQ_ERR_SHAPE;
  if (N == 0) return GQ_OK;
  if (!y || (K > 0 && (!x || !q || !bs))) return GQ_ERR_NULL;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(y, out_size(out_dtype))) return GQ_ERR_ALIGN;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, 0, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_nvfp4_gemv(c, y, ep, x, q, bs, N, K, alpha));
}

int gq_nvfp4_gemv(void* y, int out_dtype, const void* x, const uint8_t* q, const uint8_t* bs,
                  int64_t N, int64_t K, float alpha, cudaStream_t stream) {
  return gq_nvfp4_gemv_ex(y, out_dtype, x, q, bs, N, K, alpha, nullptr, stream);
}

int gq_fp8_matmul_ex(void* c_out, int out_dtype, const void* a, const uint8_t* w, int64_t M,
                     int64_t N, int64_t K, float alpha, const gq_epilogue* epilogue,
                     cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (M < 0 || N < 0 || K < 0) return GQ_ERR_SHAPE;
  if (M == 0 || N == 0) return GQ_OK;
  if (!c_out || (K > 0 && (!a || !w))) return GQ_ERR_NULL;
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(c_out, 16)) return GQ_ERR_ALIGN;
  if (M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL) return GQ_ERR_TOO_LARGE;
  // K not a multiple of 16: the tensor-map coordinates reach 16 K (int32).
  if (K % 16 != 0 && K > (1LL << 27)) return GQ_ERR_TOO_LARGE;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, 0, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_fp8_gemm(c, c_out, ep, a, w, M, N, K, alpha));
}

int gq_fp8_matmul(void* c_out, int out_dtype, const void* a, const uint8_t* w, int64_t M,
                  int64_t N, int64_t K, float alpha, cudaStream_t stream) {
  return gq_fp8_matmul_ex(c_out, out_dtype, a, w, M, N, K, alpha, nullptr, stream);
}

int gq_nvfp4_matmul_ex(void* c_out, int out_dtype, const void* a, const uint8_t* q,
                       const uint8_t* bs, int64_t M, int64_t N, int64_t K, float alpha,
                       const gq_epilogue* epilogue, cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (M < 0 || N < 0 || K < 0 || K % 64 != 0) return GQ_ERR_SHAPE;
  if (M == 0 || N == 0) return GQ_OK;
  if (!c_out || (K > 0 && (!a || !q || !bs))) return GQ_ERR_NULL;
  if (!aligned(a, 16) || !aligned(q, 16) || !aligned(bs, 4) || !aligned(c_out, 16))
    return GQ_ERR_ALIGN;
  if (M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL) return GQ_ERR_TOO_LARGE;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, 0, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_nvfp4_gemm(c, c_out, ep, a, q, bs, M, N, K, alpha));
}

int gq_nvfp4_matmul(void* c_out, int out_dtype, const void* a, const uint8_t* q,
                    const uint8_t* bs, int64_t M, int64_t N, int64_t K, float alpha,
                    cudaStream_t stream) {
  return gq_nvfp4_matmul_ex(c_out, out_dtype, a, q, bs, M, N, K, alpha, nullptr, stream);
}

int gq_fp8_grouped_matmul_ex(void* c_out, int out_dtype, const void* a, const uint8_t* w,
                             const uint32_t* a_offsets, const int32_t* expert_ids,
                             const float* expert_scales, int64_t G, int64_t E,
                             int64_t max_rows_per_group, int64_t total_M, int64_t N, int64_t K,
                             const gq_epilogue* epilogue, cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (G < 0 || E < 0 || max_rows_per_group < 0 || total_M < 0 || N < 0 || K < 0 ||
      K % 16 != 0)
    return GQ_ERR_SHAPE;
  // An empty sum with a bias would need act(bias) written per active group:
  // not supported (documented).
  if (K == 0 && epilogue != nullptr && epilogue->bias != nullptr) return GQ_ERR_SHAPE;
  if (G == 0 || total_M == 0 || N == 0 || max_rows_per_group == 0) return GQ_OK;
  if (!c_out || !a_offsets || !expert_ids || (K > 0 && (!a || (E > 0 && !w))))
    return GQ_ERR_NULL;
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(c_out, 16) || !aligned(a_offsets, 4) ||
      !aligned(expert_ids, 4) || !aligned(expert_scales, 4))
    return GQ_ERR_ALIGN;
  if (G > 65535 || E > 0x7FFFFFFFLL || total_M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL ||
      K > 0x7FFFFFFFLL)
    return GQ_ERR_TOO_LARGE;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, N, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_fp8_grouped_gemm(c, c_out, ep, a, w, a_offsets, expert_ids,
                                                       expert_scales, G, E, max_rows_per_group,
                                                       total_M, N, K));
}

int gq_fp8_grouped_matmul(void* c_out, int out_dtype, const void* a, const uint8_t* w,
                          const uint32_t* a_offsets, const int32_t* expert_ids,
                          const float* expert_scales, int64_t G, int64_t E,
                          int64_t max_rows_per_group, int64_t total_M, int64_t N, int64_t K,
                          cudaStream_t stream) {
  return gq_fp8_grouped_matmul_ex(c_out, out_dtype, a, w, a_offsets, expert_ids, expert_scales, G,
                                  E, max_rows_per_group, total_M, N, K, nullptr, stream);
}

int gq_nvfp4_grouped_matmul_ex(void* c_out, int out_dtype, const void* a, const uint8_t* q,
                               const uint8_t* bs, const uint32_t* a_offsets,
                               const int32_t* expert_ids, const float* expert_scales, int64_t G,
                               int64_t E, int64_t max_rows_per_group, int64_t total_M, int64_t N,
                               int64_t K, const gq_epilogue* epilogue, cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (G < 0 || E < 0 || max_rows_per_group < 0 || total_M < 0 || N < 0 || K < 0 ||
      K % 64 != 0)
    return GQ_ERR_SHAPE;
  if (K == 0 && epilogue != nullptr && epilogue->bias != nullptr) return GQ_ERR_SHAPE;
  if (G == 0 || total_M == 0 || N == 0 || max_rows_per_group == 0) return GQ_OK;
  if (!c_out || !a_offsets || !expert_ids || (K > 0 && (!a || (E > 0 && (!q || !bs)))))
    return GQ_ERR_NULL;
  if (!aligned(a, 16) || !aligned(q, 16) || !aligned(bs, 4) || !aligned(c_out, 16) ||
      !aligned(a_offsets, 4) || !aligned(expert_ids, 4) || !aligned(expert_scales, 4))
    return GQ_ERR_ALIGN;
  if (G > 65535 || E > 0x7FFFFFFFLL || total_M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL ||
      K > 0x7FFFFFFFLL)
    return GQ_ERR_TOO_LARGE;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, N, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_nvfp4_grouped_gemm(c, c_out, ep, a, q, bs, a_offsets,
                                                         expert_ids, expert_scales, G, E,
                                                         max_rows_per_group, total_M, N, K));
}

int gq_nvfp4_grouped_matmul(void* c_out, int out_dtype, const void* a, const uint8_t* q,
                            const uint8_t* bs, const uint32_t* a_offsets, const int32_t* expert_ids,
                            const float* expert_scales, int64_t G, int64_t E,
                            int64_t max_rows_per_group, int64_t total_M, int64_t N, int64_t K,
                            cudaStream_t stream) {
  return gq_nvfp4_grouped_matmul_ex(c_out, out_dtype, a, q, bs, a_offsets, expert_ids,
                                    expert_scales, G, E, max_rows_per_group, total_M, N, K,
                                    nullptr, stream);
}

int gq_int8_quantize_rows(int8_t* q, float* scale, const void* x, int64_t M, int64_t K,
                          cudaStream_t stream) {
  if (M < 0 || K < 0) return GQ_ERR_SHAPE;
  if (M == 0) return GQ_OK;
  if (!scale || (K > 0 && (!q || !x))) return GQ_ERR_NULL;
  if (!aligned(x, 2) || !aligned(scale, 4)) return GQ_ERR_ALIGN;
  if (M > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL) return GQ_ERR_TOO_LARGE;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_int8_quantize_rows(c, q, scale, x, M, K));
}

int gq_int8_matmul_ex(void* c_out, int out_dtype, const int8_t* a, const int8_t* b,
                      const float* a_scale, const float* b_scale, int64_t M, int64_t N,
                      int64_t K, const gq_epilogue* epilogue, cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (M < 0 || N < 0 || K < 0 || K % 16 != 0) return GQ_ERR_SHAPE;
  if (M == 0 || N == 0) return GQ_OK;
  if (!c_out || !a_scale || !b_scale || (K > 0 && (!a || !b))) return GQ_ERR_NULL;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c_out, 16) || !aligned(a_scale, 4) ||
      !aligned(b_scale, 4))
    return GQ_ERR_ALIGN;
  if (M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL || K > gq::kInt8MaxK) return GQ_ERR_TOO_LARGE;
  gq::Epi ep;
  if (int s = make_epi(out_dtype, epilogue, 0, &ep)) return s;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_int8_gemm(c, c_out, ep, a, b, a_scale, b_scale, M, N, K));
}

int gq_int8_matmul(void* c_out, int out_dtype, const int8_t* a, const int8_t* b,
                   const float* a_scale, const float* b_scale, int64_t M, int64_t N, int64_t K,
                   cudaStream_t stream) {
  return gq_int8_matmul_ex(c_out, out_dtype, a, b, a_scale, b_scale, M, N, K, nullptr, stream);
}

int gq_fp8_materialize(void* out, int out_dtype, const uint8_t* w, int64_t N, int64_t K,
                       cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (N < 0 || K < 0) return GQ_ERR_SHAPE;
  if (N == 0 || K == 0) return GQ_OK;
  if (!out || !w) return GQ_ERR_NULL;
  if (!aligned(out, 16) || !aligned(w, 16)) return GQ_ERR_ALIGN;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  const int kind = out_dtype == GQ_BF16 ? gq::kOutBf16 : (out_dtype == GQ_F16 ? gq::kOutF16 : gq::kOutF32);
  return gq::launch_status(gq::launch_fp8_materialize(c, out, kind, w, N * K));
}

int gq_nvfp4_materialize(void* out, int out_dtype, const uint8_t* q, const uint8_t* bs,
                         int64_t N, int64_t K, cudaStream_t stream) {
  if (!valid_dtype(out_dtype)) return GQ_ERR_DTYPE;
  if (N < 0 || K < 0 || K % 16 != 0) return GQ_ERR_SHAPE;
  if (N == 0 || K == 0) return GQ_OK;
  if (!out || !q || !bs) return GQ_ERR_NULL;
  if (!aligned(out, 16) || !aligned(q, 16)) return GQ_ERR_ALIGN;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  const int kind = out_dtype == GQ_BF16 ? gq::kOutBf16 : (out_dtype == GQ_F16 ? gq::kOutF16 : gq::kOutF32);
  return gq::launch_status(gq::launch_nvfp4_materialize(c, out, kind, q, bs, N * K / 16));
}

int gq_probe_gemv_read_floor(int format, void* y, const uint8_t* w, const uint8_t* bs,
                             int64_t N, int64_t K, cudaStream_t stream) {
  if (format != 0 && format != 1) return GQ_ERR_DTYPE;
  if (N < 0 || K < 0 || K % 16 != 0) return GQ_ERR_SHAPE;
  if (N == 0 || K == 0) return GQ_OK;
  if (!y || !w || (format == 1 && !bs)) return GQ_ERR_NULL;
  if (!aligned(w, 16) || !aligned(y, 2)) return GQ_ERR_ALIGN;
  gq::Ctx c;
  if (int s = gq::device_ctx(stream, &c)) return s;
  return gq::launch_status(gq::launch_gemv_read_floor(c, format, y, w, bs, N, K));
}

int gq_set_wait_limit_ns(uint64_t ns) {
  gq::Ctx c;
  if (int s = gq::device_ctx(nullptr, &c)) return s;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(reinterpret_cast<uint8_t*>(c.status) + 8, &ns, sizeof(ns),
                 cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_DEVICE;
  }
  return GQ_OK;
}

int gq_device_status(uint32_t* flags, int reset) {
  gq::Ctx c;
  if (int s = gq::device_ctx(nullptr, &c)) return s;
  uint32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&v, c.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return GQ_ERR_DEVICE;
  }
  if (flags) *flags = v;
  if (reset) {
    const uint32_t zero = 0;
    if (cudaMemcpy(c.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return GQ_ERR_DEVICE;
    }
  }
  return GQ_OK;
}

}  // extern "C"
