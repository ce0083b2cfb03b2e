// Internal helpers shared by the libw8a8 translation units (not part of the
// C ABI).  Every kernel launch goes through these checks so that argument
// errors never reach the device.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "w8a8.h"  // include/, on the include path

namespace w8a8 {

constexpr int kNumSMsGB300 = 152;

constexpr int kMaxK = 32768;

// Few-row products (2 <= M <= kSkinnyMaxM, per channel) run on the weight
// stream of the matrix-vector kernel when the activation codes of the
// padded row count (2, 4 or 8 rows) fit kSkinnyMaxCodeBytes of shared
// memory; other shapes take the tensor-core GEMM.  Measured at N=10240,
// K=2560 after an L2 flush: 14 / 18 / 27 us at 2 / 4 / 8 rows against 27-31
// us for the GEMM, and 43 us at 16 rows (dp4a-bound), hence the limit of 8.
constexpr int kSkinnyMaxM = 8;
constexpr int kSkinnyMaxCodeBytes = 64 * 1024;

// Reads and clears the device-side error word that kernels with bounded
// waits set when a wait gives up (the value says which wait).
int read_and_clear_device_error(unsigned int *code);

// Device address of that word on the current device (looked up once per
// device), passed to the kernels as an argument; nullptr on failure.
unsigned int *device_error_word();

enum DeviceErrorCode : unsigned int {
  kDevErrNone = 0,
  kDevErrFullBarrier = 1,    // producer/MMA wait on a filled stage
  kDevErrEmptyBarrier = 2,   // producer wait on a freed stage
  kDevErrAccumBarrier = 3,   // epilogue wait on a finished accumulator
  kDevErrTmemEmpty = 4,      // MMA wait on a drained accumulator
  kDevErrSmemAlign = 5,      // dynamic shared memory not 1 KB aligned (kernel did nothing)
  kDevErrRowCopy = 6,        // decode kernel: bulk copy of the activation row did not land
};

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int ceil_div(long a, long b) { return static_cast<int>((a + b - 1) / b); }

// Compute capability check for the current device, cached per device.
int check_device();

// Launch-error check after a kernel launch.
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA;
}

inline int groups_of(int K, int group_size) {
  return group_size == 0 ? 1 : K / group_size;
}

inline bool valid_group_size(int K, int group_size) {
  if (group_size == 0) return true;
  if (group_size != 64 && group_size != 128) return false;
  return K % group_size == 0;
}

// ---- kernel launchers (one per translation unit) ---------------------------

// Row quantization: rows of fp16 -> int8 (qmax 127) or packed int4 (qmax 7,
// packed != nullptr), one fp32 scale per row or per group.
int launch_row_quant(const __half *x, int R, int K, int group_size, int qmax,
                     int8_t *q, uint8_t *packed, float *scale, cudaStream_t s);

// Matrix-vector products for M == 1.
int launch_gemv_w8a8(const int8_t *xq, const float *sa, const int8_t *Wq,
                     const float *sw, int N, int K, int group_size, __half *y,
                     cudaStream_t s);
int launch_gemv_w4a8(const int8_t *xq, const float *sa, const uint8_t *Wp,
                     const float *sw, int N, int K, __half *y, cudaStream_t s);
// The whole layer for one fp16 row: quantization fused into the MV kernel.
int launch_linear_mv(const __half *x, const void *W, const float *sw, int N, int K,
                     int group_size, int wbits, __half *y, cudaStream_t s);

// Few-row products: y [M, N] from INT8 codes xq [M, K] (scales sa [M]) and
// per-channel weights, 2 <= M <= kSkinnyMaxM.
bool skinny_supported(int M, int K, int group_size);
int launch_skinny(const int8_t *xq, const float *sa, const void *W, const float *sw, int M, int N,
                  int K, int wbits, __half *y, cudaStream_t s);

// The whole layer for 2 <= M <= kSkinnyMaxM fp16 rows (skinny_supported):
// quantization fused into the few-row kernel.
int launch_linear_rows(const __half *x, const void *W, const float *sw, int M, int N, int K,
                       int wbits, __half *y, cudaStream_t s);

// Row quantization writing the INT8 codes as fp16 values.
int launch_row_quant_half(const __half *x, int R, int K, int group_size, __half *qh,
                          float *scale, cudaStream_t s);

// Tensor-core GEMM.  A is int8 codes [M, K] (a_half false) or the same codes
// as fp16 values (a_half true).  acc_out != nullptr exports the exact int32
// (per-group) sums [M, N, G] instead of the fp16 output.
int launch_gemm_tc(const void *A, bool a_half, const float *sa, const void *W,
                   const float *sw, int M, int N, int K, int group_size, int wbits,
                   __half *y, int32_t *acc_out, cudaStream_t s);

// Weight-only product on the tensor cores: fp16 x [M, K] times the integer
// weight codes, float accumulation, y = fp16(acc * s_w) (per group: the
// groups' sums rescaled and added in ascending order).
int launch_gemm_weight_only(const __half *x, const void *W, const float *sw, int M, int N, int K,
                            int group_size, int wbits, __half *y, cudaStream_t s);

}  // namespace w8a8
