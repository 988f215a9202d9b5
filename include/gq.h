/*
 * gq.h -- weight-only quantized linear layer for NVIDIA GB300 (sm_103a).
 *
 *     out = alpha * x @ dequant(W)^T          (bf16 activations, fp32 accumulation)
 *
 * Two weight formats:
 *   FP8   -- float8_e4m3fn codes W[N, K], one byte per element, row-major; one
 *            per-tensor scale (weight_scale) passed as `alpha`.
 *            Source: the "fp8_gemv" kernel page (Modular API docs,
 *            kernels/linalg/matmul/gpu/apple/fp8_gemv), first paragraph and
 *            paragraph "Scale contract".
 *   NVFP4 -- packed E2M1 nibbles q[N, K/2] (byte j of a row holds element 2j in
 *            its low nibble and element 2j+1 in its high nibble) plus
 *            float8_e4m3fn block scales bs[N, K/16], one per 16 consecutive
 *            elements of a row; the per-tensor second scale (weight_scale_2)
 *            is passed as `alpha`.  Source: the "fp4_matmul" kernel page
 *            (kernels/linalg/matmul/gpu/apple/fp4_matmul), first paragraph.
 * And the W8A8 int8 sibling method of the "int8_matmul" page
 * (gq_int8_quantize_rows, gq_int8_matmul): int8 activations and weights with
 * per-row and per-column scales.
 *
 * Common conventions for every entry point below
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller, dense row-major, and must stay valid until the work
 *     queued on `stream` has finished.  The library allocates nothing and
 *     keeps no pointer after the call returns.
 *   - Work is queued on `stream` (0 = the legacy default stream); the call does
 *     not synchronize.  Argument checks run on the host before anything is
 *     queued; a non-zero status means nothing was queued.
 *   - Activations are bfloat16 bit patterns.  Outputs are float32, bfloat16 or
 *     binary16 (`out_dtype`; the "Matmul2dFp8" struct page lists the same three
 *     for c_type), converted from the fp32 result with round-to-nearest-even.
 *   - `alpha` multiplies the fp32 sum once, before the output conversion
 *     (alpha = 1 gives the raw product).  Because a scalar factors out of the
 *     sum this equals folding the scale after the matmul.
 *   - Pointer alignment: 16 bytes for every tensor pointer (weights,
 *     activations, outputs); block scales need 1 byte.  Odd K is allowed for
 *     the FP8 GEMV (it picks a narrower load width) and the FP8 GEMM (rows
 *     staged by residue class); see each call.
 *   - Zero-sized M or N: nothing is queued, GQ_OK.  K = 0: outputs are written
 *     as alpha * 0 (through the epilogue, when there is one).
 *   - Results are deterministic: a given call on given inputs returns the same
 *     bits every time (fixed summation order, no atomics).
 *   - Every wait inside the kernels is bounded; a wait that runs out records a
 *     code in a per-device status word (gq_device_status) and the kernel
 *     returns instead of hanging.
 */
#ifndef GQ_H_
#define GQ_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQ_OK = 0,
  GQ_ERR_NULL = 1,      /* a required pointer is NULL                         */
  GQ_ERR_SHAPE = 2,     /* a size is negative or violates a format rule       */
  GQ_ERR_ALIGN = 3,     /* a pointer is not aligned as required               */
  GQ_ERR_DTYPE = 4,     /* unknown output dtype                               */
  GQ_ERR_DEVICE = 5,    /* current device is not sm_103 or cannot be queried  */
  GQ_ERR_LAUNCH = 6,    /* the kernel launch failed (cudaGetLastError)        */
  GQ_ERR_TOO_LARGE = 7, /* a size exceeds what the kernel supports            */
  GQ_ERR_EPILOGUE = 8   /* unknown activation or bias dtype in a gq_epilogue  */
} gq_status;

typedef enum { GQ_F32 = 0, GQ_BF16 = 1, GQ_F16 = 2 } gq_dtype;

/*
 * Fused epilogue (the optional elementwise epilogue of the tiled matmul,
 * "Matmul2dFp8" struct page, parameter elementwise_lambda_fn: a function of
 * the output coordinate (row, col) and the computed value, applied where the
 * result is stored).  The C ABI takes the form a linear layer uses:
 *
 *     out[m, n] = act(alpha * acc[m, n] + bias[n])
 *
 * then the output conversion.  The grouped product takes a bias row per
 * expert: bias[e, n] for the rows of a group whose expert is e (rows of a
 * group with expert id -1 stay zero, no epilogue).
 *   bias        device pointer to N elements ([E, N] for the grouped call) of
 *               type bias_dtype (GQ_F32, GQ_BF16 or GQ_F16), aligned to the
 *               element size; NULL for no bias.
 *   activation  GQ_ACT_NONE, GQ_ACT_RELU (max(v, 0); NaN stays NaN),
 *               GQ_ACT_SILU (v / (1 + exp(-v))) or GQ_ACT_GELU_TANH
 *               (0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))), evaluated in
 *               fp32 with the CUDA math library.
 * A NULL gq_epilogue pointer is the plain product (no bias, no activation).
 * Unknown codes return GQ_ERR_EPILOGUE; a misaligned bias GQ_ERR_ALIGN.
 */
typedef enum {
  GQ_ACT_NONE = 0,
  GQ_ACT_RELU = 1,
  GQ_ACT_SILU = 2,
  GQ_ACT_GELU_TANH = 3
} gq_activation;

typedef struct gq_epilogue {
  const void* bias;
  int bias_dtype;
  int activation;
} gq_epilogue;

/*
 * Process-wide launch options (default 0).
 *
 * The GEMV entry points (gq_fp8_gemv, gq_nvfp4_gemv and their _ex forms)
 * and the few-row GEMM (gq_fp8_matmul / gq_nvfp4_matmul with M <= 128)
 * always launch their kernel as a programmatic dependent of the previous
 * kernel in the stream; by default every thread waits for that kernel to
 * finish (and its writes to become visible) before it reads or writes any
 * global memory, so stream order is unchanged and only the launch gap (and,
 * for the GEMM, its set-up) is hidden.  Before that wait a GEMV CTA issues
 * an L2 prefetch of its first weight bytes: a prefetch returns no data to
 * the kernel (L2 is coherent), so it does not change what is read.
 *
 * GQ_LAUNCH_OVERLAP_WEIGHT_READS: each GEMV thread, and the few-row GEMM's
 * weight producer, issue their weight loads before that wait; activations
 * are read and outputs written only after it.  The weight stream then
 * overlaps the tail of the kernel before, which is what a decode loop over
 * layers with fixed weights wants.  Only set it when no kernel issued just
 * before such a call writes its weight buffers: those reads are not ordered
 * after the previous kernel.  Activations and outputs always are.
 * Not a citation of the pages: a GB300 launch option.
 * gq_set_launch_flags returns GQ_ERR_SHAPE for unknown bits.
 */
#define GQ_LAUNCH_OVERLAP_WEIGHT_READS 1u
/*
 * GQ_LAUNCH_TEST_STALL_PRODUCER (tests only; never set it for real work):
 * the persistent tensor-core GEMM (FP8 and NVFP4 with M > 128, FP8 with any
 * K, W8A8, grouped; not the few-row, M <= 128 split-K or GEMV kernels)
 * launches with its copy producer idle, so
 * no shared-memory stage ever fills, nothing asynchronous is issued, and every
 * bounded wait of the kernel runs out: the call returns, the output is left
 * unwritten, and gq_device_status reports the timed-out waits.  Use it with a
 * short gq_set_wait_limit_ns to exercise that failure path without a fault.
 * Not a citation of the pages.
 */
#define GQ_LAUNCH_TEST_STALL_PRODUCER 2u
int gq_set_launch_flags(uint32_t flags);
uint32_t gq_get_launch_flags(void);

/* Human-readable name of a gq_status value (static string). */
const char* gq_status_str(int status);

/* Library version, e.g. "gq 0.1.0 sm_103a". */
const char* gq_version(void);

/*
 * FP8 GEMV (M = 1 decode).  y[n] = alpha * sum_k x[k] * e4m3(w[n, k]).
 * Source: "fp8_gemv" page -- enqueue_apple_fp8_gemv and fp8_gemv_kernel (one
 * warp per output, lanes striding K, fp32 FMA, warp sum, narrow tail).
 *   y      [N]    out_dtype
 *   x      [K]    bfloat16
 *   w      [N, K] float8_e4m3fn codes
 * Any K >= 0.  Pointer alignment: 16 bytes gives the widest loads; less is
 * accepted (the load width drops to what K and the pointers allow).
 */
int gq_fp8_gemv(void* y, int out_dtype, const void* x, const uint8_t* w,
                int64_t N, int64_t K, float alpha, cudaStream_t stream);
/* The same with a fused epilogue (see gq_epilogue; NULL = gq_fp8_gemv). */
int gq_fp8_gemv_ex(void* y, int out_dtype, const void* x, const uint8_t* w,
                   int64_t N, int64_t K, float alpha, const gq_epilogue* epilogue,
                   cudaStream_t stream);

/*
 * NVFP4 GEMV (M = 1).  y[n] = alpha * sum_k x[k] * e2m1(q[n, k]) * e4m3(bs[n, k/16]).
 * Source: "fp4_matmul" page (weight layout); the "fp8_gemv" page names this
 * kernel as the FP4 sibling of its GEMV (nibble unpack, E2M1 decode, per-16
 * FP8 block scale).
 *   y [N] (out_dtype), x [K] bfloat16, q [N, K/2] uint8, bs [N, K/16] uint8.
 * K % 16 == 0 (GQ_ERR_SHAPE otherwise).  q, x, y 16-byte aligned.
 */
int gq_nvfp4_gemv(void* y, int out_dtype, const void* x, const uint8_t* q,
                  const uint8_t* bs, int64_t N, int64_t K, float alpha,
                  cudaStream_t stream);
/* The same with a fused epilogue (see gq_epilogue; NULL = gq_nvfp4_gemv). */
int gq_nvfp4_gemv_ex(void* y, int out_dtype, const void* x, const uint8_t* q,
                     const uint8_t* bs, int64_t N, int64_t K, float alpha,
                     const gq_epilogue* epilogue, cudaStream_t stream);

/*
 * FP8 GEMM (M >= 1).  c[m, n] = alpha * sum_k a[m, k] * e4m3(w[n, k]).
 * Source: "fp8_gemv" page -- enqueue_apple_fp8_matmul (raw W8A16 matmul);
 * "Matmul2dFp8" page (bf16 A x fp8 B -> fp32, c_type output).
 *   c [M, N] (out_dtype), a [M, K] bfloat16, w [N, K] float8_e4m3fn.
 * M, N, K arbitrary.  Pointers 16-byte aligned.  With K % 16 == 0 the
 * operands are staged by the tensor memory accelerator; otherwise their rows
 * are not 16-byte strided: they are staged by residue class (rows 8 apart in
 * a, 16 apart in w are 16-byte strided) and realigned in shared memory (the
 * "fp4_matmul" page's K tail, generalised to any K); then K <= 2^27
 * (GQ_ERR_TOO_LARGE otherwise).
 */
int gq_fp8_matmul(void* c, int out_dtype, const void* a, const uint8_t* w,
                  int64_t M, int64_t N, int64_t K, float alpha,
                  cudaStream_t stream);
/* The same with a fused epilogue (see gq_epilogue; NULL = gq_fp8_matmul). */
int gq_fp8_matmul_ex(void* c, int out_dtype, const void* a, const uint8_t* w,
                     int64_t M, int64_t N, int64_t K, float alpha,
                     const gq_epilogue* epilogue, cudaStream_t stream);

/*
 * NVFP4 GEMM (M >= 1).  c = alpha * a @ dequant(q, bs)^T.
 * Source: "fp4_matmul" page -- enqueue_apple_fp4_matmul and AppleM5Fp4MatMul
 * (packed weight stays packed in memory; each weight tile is dequantized to
 * bf16 once into shared memory and fed to a dense bf16 MMA).
 *   c [M, N] (out_dtype), a [M, K] bf16, q [N, K/2] uint8, bs [N, K/16] uint8.
 * K % 64 == 0 (GQ_ERR_SHAPE otherwise).  Pointers 16-byte aligned, bs 4-byte.
 */
int gq_nvfp4_matmul(void* c, int out_dtype, const void* a, const uint8_t* q,
                    const uint8_t* bs, int64_t M, int64_t N, int64_t K,
                    float alpha, cudaStream_t stream);
/* The same with a fused epilogue (see gq_epilogue; NULL = gq_nvfp4_matmul). */
int gq_nvfp4_matmul_ex(void* c, int out_dtype, const void* a, const uint8_t* q,
                       const uint8_t* bs, int64_t M, int64_t N, int64_t K,
                       float alpha, const gq_epilogue* epilogue, cudaStream_t stream);

/*
 * Grouped (MoE) FP8 GEMM.  For every group z in [0, G):
 *   rows r in [a_offsets[z], a_offsets[z+1]):
 *     c[r, :] = 0                                     if expert_ids[z] == -1
 *     c[r, :] = s_e * a[r, :] @ e4m3(w[e, :, :])^T    with e = expert_ids[z],
 *               s_e = expert_scales[e] (1 when expert_scales is NULL)
 * Source: "Matmul2dFp8" page, method run_grouped (ragged groups from
 * a_offsets, empty groups do nothing, expert id -1 writes zeros, the
 * per-expert scale folded after the product).
 *   c             [total_M, N] (out_dtype)
 *   a             [total_M, K] bfloat16
 *   w             [E, N, K]    float8_e4m3fn, one weight per expert
 *   a_offsets     [G + 1]      uint32, device memory
 *   expert_ids    [G]          int32, device memory
 *   expert_scales [E]          float32, device memory, or NULL (raw)
 *   max_rows_per_group         an upper bound on a_offsets[z+1] - a_offsets[z]
 * Device-side data is not checked on the host (that would need a sync); the
 * kernel treats it defensively: an id outside [0, E) other than -1 is
 * treated as -1, a group with a_offsets[z+1] <= a_offsets[z] is empty, rows
 * outside [0, total_M) are never read or written, rows that no group covers
 * are left untouched, and rows beyond max_rows_per_group in a group are not
 * computed (out of contract).  K % 16 == 0.
 */
int gq_fp8_grouped_matmul(void* c, int out_dtype, const void* a,
                          const uint8_t* w, const uint32_t* a_offsets,
                          const int32_t* expert_ids, const float* expert_scales,
                          int64_t G, int64_t E, int64_t max_rows_per_group,
                          int64_t total_M, int64_t N, int64_t K,
                          cudaStream_t stream);
/* The same with a fused epilogue; its bias is [E, N] (row e for expert e).
 * K = 0 with a bias returns GQ_ERR_SHAPE.  NULL = gq_fp8_grouped_matmul. */
int gq_fp8_grouped_matmul_ex(void* c, int out_dtype, const void* a,
                             const uint8_t* w, const uint32_t* a_offsets,
                             const int32_t* expert_ids, const float* expert_scales,
                             int64_t G, int64_t E, int64_t max_rows_per_group,
                             int64_t total_M, int64_t N, int64_t K,
                             const gq_epilogue* epilogue, cudaStream_t stream);

/*
 * Grouped (MoE) NVFP4 GEMM: gq_fp8_grouped_matmul's groups with NVFP4 experts.
 * Source: the "Matmul2dFp8" page, method run_grouped (the grouped schedule),
 * and the "fp4_matmul" page (the NVFP4 weight): for every group z, rows
 * r in [a_offsets[z], a_offsets[z+1]):
 *     c[r, :] = 0                                              if expert_ids[z] == -1
 *     c[r, :] = s_e * a[r, :] @ (e2m1(q[e]) * e4m3(bs[e]))^T   with e = expert_ids[z],
 *               s_e = expert_scales[e] (the expert's second scale; 1 when NULL)
 *   c [total_M, N] (out_dtype), a [total_M, K] bfloat16,
 *   q [E, N, K/2] uint8 (packed, low nibble first), bs [E, N, K/16] uint8,
 *   a_offsets, expert_ids, expert_scales, max_rows_per_group: as in
 *   gq_fp8_grouped_matmul (same defensive treatment of device-side data).
 * K % 64 == 0.  Pointers 16-byte aligned, bs 4-byte.
 */
int gq_nvfp4_grouped_matmul(void* c, int out_dtype, const void* a, const uint8_t* q,
                            const uint8_t* bs, const uint32_t* a_offsets,
                            const int32_t* expert_ids, const float* expert_scales,
                            int64_t G, int64_t E, int64_t max_rows_per_group,
                            int64_t total_M, int64_t N, int64_t K, cudaStream_t stream);
/* The same with a fused epilogue; its bias is [E, N].  K = 0 with a bias
 * returns GQ_ERR_SHAPE.  NULL = gq_nvfp4_grouped_matmul. */
int gq_nvfp4_grouped_matmul_ex(void* c, int out_dtype, const void* a, const uint8_t* q,
                               const uint8_t* bs, const uint32_t* a_offsets,
                               const int32_t* expert_ids, const float* expert_scales,
                               int64_t G, int64_t E, int64_t max_rows_per_group,
                               int64_t total_M, int64_t N, int64_t K,
                               const gq_epilogue* epilogue, cudaStream_t stream);

/*
 * W8A8 int8, activation side: per-row symmetric absmax quantization.
 * Source: the "int8_matmul" page, enqueue_apple_int8_quantize_activation
 * (A quantized online, one fp32 scale per row, scale = absmax / 127).
 *     scale[m] = max_k |x[m, k]| / 127                      (float32 division)
 *     q[m, k]  = clamp(rint(x[m, k] / scale[m]), -127, 127) (float32 division,
 *                round half to even); a row of zeros: scale 0, codes 0.
 *   x [M, K] bfloat16 (2-byte aligned; finite values), q [M, K] int8,
 *   scale [M] float32 (4-byte aligned).  Any M, K; rows that are 16-byte
 *   aligned with K % 16 == 0 and K <= 8192 are read once, others twice.
 */
int gq_int8_quantize_rows(int8_t* q, float* scale, const void* x, int64_t M, int64_t K,
                          cudaStream_t stream);

/*
 * W8A8 int8 GEMM.  Source: the "int8_matmul" page, enqueue_apple_int8_matmul:
 *     acc[m, n] = sum_k a[m, k] * b[n, k]           (exact integer products)
 *     c[m, n]   = (acc * a_scale[m]) * b_scale[n]   (float32, each product
 *                 rounded once), then the epilogue (bias after the dequant,
 *                 activation), then the output conversion.
 *   c [M, N] (out_dtype), a [M, K] int8, b [N, K] int8 (one row per output
 *   column), a_scale [M], b_scale [N] float32.  K % 16 == 0 and
 *   K <= 130560 (GQ_ERR_TOO_LARGE beyond: |acc| then stays inside int32 for
 *   any codes).  a, b, c 16-byte aligned; scales 4-byte aligned.
 * acc is the exact int32 sum for every input, as on the page.  GB300 has no
 * int8 tensor-core instruction on sm_103a (tcgen05 kind::i8 is not
 * available there), so the sums run on binary16 tensor-core products: both
 * operands' codes are widened exactly to binary16, every product is an
 * integer of magnitude at most 2^14, the products of each chunk of at most
 * 1024 K are summed in float32 (every partial sum is an integer of magnitude
 * at most 2^24, so exact), and the chunks are added in int32.  With small M,
 * K may be split over a thread-block cluster of CTAs whose int32 partials
 * are added exactly.  acc is converted to float32 with round-to-nearest-even.
 */
int gq_int8_matmul(void* c, int out_dtype, const int8_t* a, const int8_t* b,
                   const float* a_scale, const float* b_scale, int64_t M, int64_t N,
                   int64_t K, cudaStream_t stream);
/* The same with a fused epilogue (see gq_epilogue; NULL = gq_int8_matmul). */
int gq_int8_matmul_ex(void* c, int out_dtype, const int8_t* a, const int8_t* b,
                      const float* a_scale, const float* b_scale, int64_t M, int64_t N,
                      int64_t K, const gq_epilogue* epilogue, cudaStream_t stream);

/*
 * FP8 materialize: out[n, k] = e4m3(w[n, k]) as float32, bfloat16 or binary16,
 * exact (every E4M3 value is representable in all three), no scale applied.
 * Source: "fp8_gemv" page -- enqueue_fp8_materialize / fp8_materialize_kernel.
 *   out [N, K] (out_dtype), w [N, K].
 */
int gq_fp8_materialize(void* out, int out_dtype, const uint8_t* w,
                       int64_t N, int64_t K, cudaStream_t stream);

/*
 * NVFP4 materialize: out[n, k] = e2m1(q[n, k]) * e4m3(bs[n, k/16]), exact in
 * float32, bfloat16 and binary16 (the product has at most 6 significant bits
 * and lies in [2^-10, 2688]), no per-tensor scale applied.  Source: "fp4_matmul" page (weight layout); the
 * NVFP4 counterpart of the FP8 materialize.
 *   out [N, K] (out_dtype), q [N, K/2], bs [N, K/16].  K % 16 == 0.
 */
int gq_nvfp4_materialize(void* out, int out_dtype, const uint8_t* q,
                         const uint8_t* bs, int64_t N, int64_t K,
                         cudaStream_t stream);

/*
 * Status word of the current device: bit flags recorded by kernels whose
 * bounded waits ran out (0 = none).  Synchronizes the device.  If `reset` is
 * non-zero the word is cleared afterwards.  Returns GQ_OK or GQ_ERR_DEVICE.
 */
int gq_device_status(uint32_t* flags, int reset);

/*
 * Measurement probe (not a citation of the pages): the HBM floor of the
 * GEMVs' launch shapes.  Runs the FP8 (format 0; w [N, K], K % 16 == 0,
 * 16-byte aligned) or NVFP4 (format 1; w = q [N, K/2], bs [N, K/16]) GEMV
 * kernel with its grid, CTA shape, L2 prefetch, dependent launch and weight
 * loads unchanged but the decode and the arithmetic left out: it reads every
 * weight and block-scale byte once and writes one checksum value per row to
 * y ([N] bfloat16, caller-owned; an integer in [0, 128]).  The time of a call is what the GEMV of
 * the same shape would take if its arithmetic were free.  Returns GQ_OK or a
 * GQ_ERR code (format: GQ_ERR_DTYPE).
 */
int gq_probe_gemv_read_floor(int format, void* y, const uint8_t* w, const uint8_t* bs,
                             int64_t N, int64_t K, cudaStream_t stream);

/*
 * How long a bounded in-kernel wait of the current device polls before it
 * gives up (records its bit in the status word and lets the kernel unwind):
 * `ns` nanoseconds, or the default of 2 s when ns == 0.  Applies to kernels
 * launched after the call returns; synchronizes the device.  Meant for tests
 * of the failure path (with GQ_LAUNCH_TEST_STALL_PRODUCER); a limit shorter
 * than a kernel's real waits makes it give up on valid work.  Not a citation
 * of the pages.  Returns GQ_OK or GQ_ERR_DEVICE.
 */
int gq_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* GQ_H_ */
