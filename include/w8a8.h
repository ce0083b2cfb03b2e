/*
 * w8a8.h -- C ABI of libw8a8, the GB300 (sm_103a) W8A8 / W4A8 quantized
 * linear layer.
 *
 * The method: "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다"
 * (molayo1419.me), section "INT8 TensorOps 커널 설계", describes a four-step
 * pipeline -- (1) a min/max reduction that gives each activation row its
 * scale, (2) a streaming fp16 -> INT8 mapping, (3) an INT8 x INT8 GEMM that
 * accumulates in INT32, (4) a rescale of the INT32 result by the product of
 * the activation and weight scales into fp16 -- and section
 * "입도(Granularity)" adds per-group scales (64 or 128 elements) that need
 * grouped dequantization during accumulation.  "cider 소개"
 * (discuss.pytorch.kr), section "cider의 양자화 모드와 적용 가능한 영역",
 * fixes the modes: symmetric INT8 weights, per-token INT8 activations,
 * per-channel or per-group (gs 128 / 64) scales, and W4A8 with INT4 weights
 * packed in uint8 and unpacked before the INT8 matmul; its section
 * "cider 설치와 사용법" names quantize_weight_int8 / pack_weight_int4 and
 * the seq_len rule of CiderLinear (seq_len > 1: GEMM, seq_len == 1: INT8
 * matrix-vector kernel).
 *
 * Conventions for every entry point below
 * ---------------------------------------
 *  - Shapes: x [M, K] fp16 row-major (K contiguous); W [N, K] row-major
 *    (out_features x in_features); y = x . W^T, [M, N] fp16 row-major.
 *    G = K / group_size groups along K (G = 1 when group_size == 0).
 *  - fp16 buffers are IEEE binary16 bit patterns (w8a8_half).
 *  - Every pointer is a DEVICE pointer on the current CUDA device, owned by
 *    the caller.  The library allocates no device memory and keeps no
 *    pointer after a call returns.
 *  - The library caches per-device state (function attributes, the SM
 *    count, the device addresses of its own device variables) on the first
 *    call on each device; the caches are thread-safe.  Do not use the
 *    library on a device after cudaDeviceReset() in the same process: the
 *    cached addresses would be stale.
 *  - Matrix pointers (x, W, Wq, Wp, xq, y, acc, workspace) must be 16-byte
 *    aligned, scale pointers 4-byte aligned, and K a multiple of 16 (32 for
 *    packed INT4 weights), else W8A8_ERR_MISALIGNED.  K is at most 32768
 *    (else W8A8_ERR_INVALID_ARG); this also keeps every INT32 sum in range
 *    (127 * 127 * 32768 < 2^31).
 *  - group_size is 0 (one scale per row: per-token activations,
 *    per-output-channel weights), 64 or 128; K % group_size must be 0.
 *  - M == 0 or N == 0 is an empty problem: the call returns W8A8_OK and
 *    launches nothing.  Negative sizes and K <= 0 are W8A8_ERR_INVALID_ARG.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are detected on the host before any
 *    launch, and then no output is touched.
 *  - Inputs must be finite; the result of a NaN or Inf input is unspecified.
 *  - Rounding: scale = absmax / qmax with one IEEE fp32 division; q =
 *    clamp(rint(x / scale), -qmax, qmax) with an IEEE fp32 division and
 *    ties to even; a group whose absmax is 0 gets scale 0 and q 0; -128 is
 *    never produced.  Dequant: per channel y = fp16_rn((float)acc *
 *    (s_a * s_w)); per group y = fp16_rn(sum over g of (float)acc_g *
 *    (s_a,g * s_w,g)), INT32 partials per group.
 */
#ifndef W8A8_H
#define W8A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t w8a8_half;   /* IEEE binary16 bit pattern */
typedef void *w8a8_stream_t;  /* a cudaStream_t */

/* Status codes returned by every call. */
#define W8A8_OK 0
#define W8A8_ERR_INVALID_ARG 1        /* null pointer, bad size, bad group_size */
#define W8A8_ERR_MISALIGNED 2         /* pointer not 16-byte aligned, K % 16 */
#define W8A8_ERR_UNSUPPORTED_DEVICE 3 /* current device is not compute 10.3 */
#define W8A8_ERR_CUDA 4               /* a CUDA runtime call or launch failed */
#define W8A8_ERR_TIMEOUT 5            /* a bounded device-side wait gave up */
#define W8A8_ERR_WORKSPACE 6          /* workspace too small */

/* 1 if the current CUDA device is a compute-capability 10.3 GPU (GB300)
 * that this library's kernels were built for, else 0.  The analogue of the
 * SDK's is_available() ("cider 설치와 사용법"). */
int w8a8_is_available(void);

/* Static, human-readable name of a status code. */
const char *w8a8_status_string(int status);

/* Reads and clears the device-side error word that the kernels set when a
 * bounded wait on the tensor-core pipeline gives up, or when a GEMM kernel
 * finds its shared memory not 1 KB aligned and returns without doing
 * anything (both leave the outputs of that call undefined).  Synchronizes
 * `stream`.  Returns W8A8_OK, W8A8_ERR_TIMEOUT (for either cause) or
 * W8A8_ERR_CUDA. */
int w8a8_check_status(w8a8_stream_t stream);

/* Offline INT8 weight quantization ("cider 설치와 사용법":
 * quantize_weight_int8(W) -> (w_int8, scale); mode table: symmetric INT8).
 *   W        fp16 [N, K]
 *   Wq       int8 [N, K]        (out)
 *   scale_w  fp32 [N, G]        (out) absmax / 127 per row (per group)
 * group_size 0 = per output channel. */
int quantize_weight_int8(const w8a8_half *W, int N, int K, int group_size,
                         int8_t *Wq, float *scale_w, w8a8_stream_t stream);

/* Offline INT4 weight quantization and packing ("cider 설치와 사용법":
 * pack_weight_int4(W) -> (packed, scale); mode table: W4A8, INT4 packed in
 * uint8).  Per output channel: s4 = absmax / 7, q4 = clamp(rint(W / s4),
 * -7, 7); byte j of row n holds q4[n, 2j] in its low nibble and
 * q4[n, 2j+1] in its high nibble, both two's complement.
 *   W        fp16 [N, K], K % 32 == 0
 *   Wp       uint8 [N, K/2]     (out)
 *   scale_w  fp32 [N]           (out) */
int pack_weight_int4(const w8a8_half *W, int N, int K, uint8_t *Wp,
                     float *scale_w, w8a8_stream_t stream);

/* Online per-token activation quantization ("INT8 TensorOps 커널 설계",
 * steps 1-2; mode table: INT8 per token).
 *   x        fp16 [M, K]
 *   xq       int8 [M, K]        (out)
 *   scale_a  fp32 [M, G]        (out) absmax / 127 per row (per group) */
int quantize_act_per_token(const w8a8_half *x, int M, int K, int group_size,
                           int8_t *xq, float *scale_a, w8a8_stream_t stream);

/* W8A8 GEMM with fused dequant ("INT8 TensorOps 커널 설계" steps 3-4;
 * "입도(Granularity)" for group_size > 0).  Exact INT32 (per-group) sums,
 * then the fp32 rescale and one fp16 rounding.
 *   xq       int8 [M, K],  scale_a fp32 [M, G]
 *   Wq       int8 [N, K],  scale_w fp32 [N, G]
 *   y        fp16 [M, N]        (out)
 * Any M >= 1 is accepted (M == 1 runs the matrix-vector kernel). */
int w8a8_gemm(const int8_t *xq, const float *scale_a, const int8_t *Wq,
              const float *scale_w, int M, int N, int K, int group_size,
              w8a8_half *y, w8a8_stream_t stream);

/* W8A8 matrix-vector product for decode (the SDK's INT8 MV kernel for
 * seq_len == 1, "cider 소개", section "cider의 동작 방식과 자동 경로 선택";
 * per channel or per group).  Same arguments as w8a8_gemm; M must be 1 (else
 * W8A8_ERR_INVALID_ARG).
 * Ordering: the matrix-vector kernel is launched with programmatic stream
 * serialization, and it may start reading Wq (only Wq) before the previous
 * kernel on the stream has finished when that kernel lets its dependents
 * start early (executes griddepcontrol.launch_dependents).  Do not write Wq
 * in such a kernel right before this call; the library's own kernels that
 * write weights never let dependents start early.  The same holds for
 * w4a8_gemm and linear with M == 1. */
int w8a8_mv(const int8_t *xq, const float *scale_a, const int8_t *Wq,
            const float *scale_w, int M, int N, int K, int group_size,
            w8a8_half *y, w8a8_stream_t stream);

/* W4A8 GEMM ("cider 설치와 사용법": w4a8_linear; mode table: W4A8,
 * unpack -> INT8 matmul).  Per-channel INT4 weights packed as
 * pack_weight_int4 writes them, per-token INT8 activations.
 *   xq int8 [M, K], scale_a fp32 [M]; Wp uint8 [N, K/2], scale_w fp32 [N];
 *   y fp16 [M, N] (out); K % 32 == 0.  M == 1 runs the W4A8 matrix-vector
 *   kernel. */
int w4a8_gemm(const int8_t *xq, const float *scale_a, const uint8_t *Wp,
              const float *scale_w, int M, int N, int K, w8a8_half *y,
              w8a8_stream_t stream);

/* quantize_act_per_token with the INT8 codes written as fp16 values (every
 * code in [-127, 127] is an fp16 integer exactly): the operand format the
 * tensor-core GEMM reads without converting, which linear() uses for M > 1.
 *   x        fp16 [M, K]
 *   xq_h     fp16 [M, K]        (out) the codes q, as fp16
 *   scale_a  fp32 [M, G]        (out)
 * Ordering: the kernel lets the next kernel on the stream start early
 * (griddepcontrol.launch_dependents), which only matters to a kernel
 * launched with programmatic stream serialization; the library's GEMM is,
 * and it waits for this kernel to finish before reading any input. */
int quantize_act_per_token_h(const w8a8_half *x, int M, int K, int group_size,
                             w8a8_half *xq_h, float *scale_a, w8a8_stream_t stream);

/* The GEMM of w8a8_gemm (wbits 8) or w4a8_gemm (wbits 4, group_size 0) with
 * the activation codes given as fp16 values, as quantize_act_per_token_h
 * writes them.  Codes outside [-127, 127] or not integral are outside the
 * contract.  Always the tensor-core GEMM, for any M >= 1.
 *   xq_h fp16 [M, K], scale_a fp32 [M, G]; Wq int8 [N, K] or packed uint8
 *   [N, K/2]; scale_w fp32 [N, G]; y fp16 [M, N] (out)
 * The GEMM (any M, every GEMM entry point) is launched with programmatic
 * stream serialization: its set-up may overlap the previous kernel on the
 * stream, and it reads no input before that kernel has finished. */
int w8a8_gemm_h(const w8a8_half *xq_h, const float *scale_a, const void *Wq,
                const float *scale_w, int M, int N, int K, int group_size, int wbits,
                w8a8_half *y, w8a8_stream_t stream);

/* Bytes of workspace that linear() needs for M rows of K activations: the
 * activation codes (fp16 values for M > 1, INT8 for M == 1) and their fp32
 * scales, each region 256-byte aligned. */
size_t w8a8_linear_workspace_bytes(int M, int K, int group_size);

/* The whole layer, CiderLinear's forward ("cider 소개", section "cider의
 * 동작 방식과 자동 경로 선택": seq_len > 1 -> INT8 GEMM, seq_len == 1 ->
 * INT8 MV kernel).  M == 1: one kernel quantizes the row and runs the
 * matrix-vector product with the fused dequant.  2 <= M <= 8, per channel,
 * with the codes of the rows (padded to 2, 4 or 8) within 64 KB: one kernel
 * quantizes the rows and runs the few-row product on the same weight
 * stream.  In both, the workspace is checked but not written (see w8a8_mv
 * for the ordering rule of those kernels).  Otherwise: quantize x per token
 * into the workspace (quantize_act_per_token_h), then the GEMM
 * (w8a8_gemm_h) with the fused dequant.  Same quantization rule everywhere.
 *   x        fp16 [M, K]
 *   Wq       int8 [N, K] (wbits 8) or packed uint8 [N, K/2] (wbits 4)
 *   scale_w  fp32 [N, G] (wbits 4 requires group_size 0)
 *   workspace device buffer of at least w8a8_linear_workspace_bytes(M, K,
 *            group_size) bytes, 256-byte aligned, else W8A8_ERR_WORKSPACE
 *   y        fp16 [M, N] (out) */
int linear(const w8a8_half *x, const void *Wq, const float *scale_w, int M,
           int N, int K, int group_size, int wbits, void *workspace,
           size_t ws_bytes, w8a8_half *y, w8a8_stream_t stream);

/* linear() with no workspace argument, for callers that cannot allocate
 * device memory on their execution path (for example a serving runtime's
 * per-request path, where cudaMalloc may synchronize the device and fail
 * under memory pressure, or a plugin inside a host framework that owns all
 * device memory and exposes no allocator).  No counterpart on the method's
 * pages: an addition of this library.
 *   Arguments as linear(), minus workspace / ws_bytes.  The workspace is a
 *   fixed 8 MiB array in the library's device memory (held by every GPU that
 *   loads the library until the process exits); a problem whose
 *   w8a8_linear_workspace_bytes(M, K, group_size) exceeds 8 MiB returns
 *   W8A8_ERR_WORKSPACE and touches nothing.  Calls no allocator.
 *   All calls on a device share the array: calls whose kernels overlap on
 *   the GPU (unordered streams) race; calls on one stream are safe.  The
 *   first call on a device looks up the array's address, once per device;
 *   make it before any stream capture begins. */
int linear_noalloc(const w8a8_half *x, const void *Wq, const float *scale_w, int M,
                   int N, int K, int group_size, int wbits, w8a8_half *y,
                   w8a8_stream_t stream);

/* The weight-only product the method is measured against (W8A16 / W4A16:
 * "Apple Silicon의 AI 한계치는 당신의 생각보다 높습니다", the section on
 * MLX's weight-only quantization -- integer weights dequantized and
 * multiplied with fp16 activations; "cider 소개", mode table, W8A16 /
 * W4A16 rows, and the w8a16 / w4a16 columns of the latency table).  The
 * activations stay fp16: y = x . (q * s_w)^T, accumulated in fp32 on the
 * tensor cores (the integer codes are exact fp16 operands), then scaled by
 * s_w (per group: each group's sum scaled and added in ascending order) and
 * rounded once to fp16.  Not bit-exact against the double-precision
 * definition: within |dy| <= 2e-3 * max|y| + one fp16 ulp.
 *   x        fp16 [M, K]
 *   Wq       int8 [N, K] (wbits 8) or packed uint8 [N, K/2] (wbits 4, as
 *            pack_weight_int4 writes them; requires group_size 0)
 *   scale_w  fp32 [N, G]
 *   y        fp16 [M, N]       (out)
 * Any M >= 1 (the tensor-core GEMM, launched like w8a8_gemm_h). */
int weight_only_gemm(const w8a8_half *x, const void *Wq, const float *scale_w, int M, int N,
                     int K, int group_size, int wbits, w8a8_half *y, w8a8_stream_t stream);

/* Test export of step 3 alone ("INT8 TensorOps 커널 설계": INT32
 * accumulation): acc[m, n, g] = sum over k in group g of xq[m, k] *
 * Wq[n, k], exact, as int32 [M, N, G], through the same tensor-core
 * contraction the GEMM uses.  wbits 4 reads packed weights [N, K/2] and
 * needs group_size 0. */
int w8a8_gemm_i32(const int8_t *xq, const void *Wq, int M, int N, int K,
                  int group_size, int wbits, int32_t *acc,
                  w8a8_stream_t stream);

/* Test hook of the failure path (the method has no counterpart): sets, for
 * the tensor-core GEMM launches that follow (every entry point that runs
 * it), the limit of its bounded device-side waits in SM clock cycles
 * (0 = the default, about 2 s) and, with skip_first_copy = 1, leaves the
 * first weight-staging copy of each CTA unissued, so that the wait for it
 * gives up: the kernel then returns early, its outputs are undefined, and
 * w8a8_check_status() reports W8A8_ERR_TIMEOUT.  No fault, trap or hang is
 * involved; the kernel still lets every copy it issued land before it
 * exits.  Process-wide; w8a8_test_set_fault(0, 0) restores normal
 * operation.  Returns W8A8_ERR_INVALID_ARG for a negative limit or a flag
 * other than 0 / 1. */
int w8a8_test_set_fault(long long wait_limit_cycles, int skip_first_copy);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_H */
