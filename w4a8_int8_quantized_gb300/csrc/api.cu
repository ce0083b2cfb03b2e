// The C ABI of libw8a8: host-side argument checks, then kernel dispatch on
// the caller's stream.  See include/w8a8.h for the contract of each call.
//
// Dispatch follows CiderLinear's rule ("cider 소개", section "cider의 성능
// 측정 결과": seq_len > 1 -> INT8 GEMM, seq_len == 1 -> INT8 MV kernel),
// applied to M, the flattened row count.
#include <mutex>

#include "common.cuh"

namespace w8a8 {

int check_device() {
  // 0 = unknown, 1 = compute 10.3, 2 = something else
  static int cache[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return W8A8_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev < 0 || dev >= 64) return W8A8_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return W8A8_ERR_UNSUPPORTED_DEVICE;
    }
    cache[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return cache[dev] == 1 ? W8A8_OK : W8A8_ERR_UNSUPPORTED_DEVICE;
}

namespace {

inline bool aligned4(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 3u) == 0;
}

inline size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Shape / group checks shared by every call.  Returns W8A8_OK, or the error.
int check_shape(long M, long N, int K, int group_size, int k_multiple) {
  if (M < 0 || N < 0 || K <= 0 || K > kMaxK) return W8A8_ERR_INVALID_ARG;
  if (!valid_group_size(K, group_size)) return W8A8_ERR_INVALID_ARG;
  if (K % k_multiple != 0) return W8A8_ERR_MISALIGNED;
  return W8A8_OK;
}

int check_ptrs16(std::initializer_list<const void *> ps) {
  for (const void *p : ps) {
    if (p == nullptr) return W8A8_ERR_INVALID_ARG;
  }
  for (const void *p : ps) {
    if (!aligned16(p)) return W8A8_ERR_MISALIGNED;
  }
  return W8A8_OK;
}

int check_ptrs4(std::initializer_list<const void *> ps) {
  for (const void *p : ps) {
    if (p == nullptr) return W8A8_ERR_INVALID_ARG;
  }
  for (const void *p : ps) {
    if (!aligned4(p)) return W8A8_ERR_MISALIGNED;
  }
  return W8A8_OK;
}

#define W8A8_TRY(expr)            \
  do {                            \
    int _st = (expr);             \
    if (_st != W8A8_OK) return _st; \
  } while (0)

inline cudaStream_t as_stream(w8a8_stream_t s) {
  return static_cast<cudaStream_t>(s);
}

int gemm_dispatch(const int8_t *xq, const float *sa, const void *W,
                  const float *sw, int M, int N, int K, int gs, int wbits,
                  __half *y, cudaStream_t s) {
  if (M == 1) {
    if (wbits == 4)
      return launch_gemv_w4a8(xq, sa, static_cast<const uint8_t *>(W), sw, N, K,
                              y, s);
    return launch_gemv_w8a8(xq, sa, static_cast<const int8_t *>(W), sw, N, K,
                            gs, y, s);
  }
  // a few rows: the weight stream of the matrix-vector kernel
  if (skinny_supported(M, K, gs)) return launch_skinny(xq, sa, W, sw, M, N, K, wbits, y, s);
  return launch_gemm_tc(xq, false, sa, W, sw, M, N, K, gs, wbits, y, nullptr, s);
}

// fp16 activation codes: the tensor-core GEMM for any M
int gemm_h_dispatch(const void *xq_h, const float *sa, const void *W, const float *sw,
                    int M, int N, int K, int gs, int wbits, __half *y, cudaStream_t s) {
  return launch_gemm_tc(xq_h, true, sa, W, sw, M, N, K, gs, wbits, y, nullptr, s);
}

}  // namespace
}  // namespace w8a8

using namespace w8a8;

extern "C" {

int w8a8_is_available(void) { return check_device() == W8A8_OK ? 1 : 0; }

const char *w8a8_status_string(int status) {
  switch (status) {
    case W8A8_OK: return "ok";
    case W8A8_ERR_INVALID_ARG: return "invalid argument";
    case W8A8_ERR_MISALIGNED: return "misaligned pointer or K";
    case W8A8_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case W8A8_ERR_CUDA: return "CUDA error";
    case W8A8_ERR_TIMEOUT: return "device-side wait timed out (or kernel did not run: shared memory misaligned)";
    case W8A8_ERR_WORKSPACE: return "workspace too small or misaligned";
    default: return "unknown status";
  }
}

int w8a8_check_status(w8a8_stream_t stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return W8A8_ERR_CUDA;
  unsigned int code = 0;
  W8A8_TRY(read_and_clear_device_error(&code));
  return code == 0 ? W8A8_OK : W8A8_ERR_TIMEOUT;
}

int quantize_weight_int8(const w8a8_half *W, int N, int K, int group_size,
                         int8_t *Wq, float *scale_w, w8a8_stream_t stream) {
  W8A8_TRY(check_shape(0, N, K, group_size, 16));
  if (N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({W, Wq}));
  W8A8_TRY(check_ptrs4({scale_w}));
  W8A8_TRY(check_device());
  return launch_row_quant(reinterpret_cast<const __half *>(W), N, K, group_size,
                          127, Wq, nullptr, scale_w, as_stream(stream));
}

int pack_weight_int4(const w8a8_half *W, int N, int K, uint8_t *Wp,
                     float *scale_w, w8a8_stream_t stream) {
  W8A8_TRY(check_shape(0, N, K, 0, 32));
  if (N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({W, Wp}));
  W8A8_TRY(check_ptrs4({scale_w}));
  W8A8_TRY(check_device());
  return launch_row_quant(reinterpret_cast<const __half *>(W), N, K, 0, 7,
                          nullptr, Wp, scale_w, as_stream(stream));
}

int quantize_act_per_token(const w8a8_half *x, int M, int K, int group_size,
                           int8_t *xq, float *scale_a, w8a8_stream_t stream) {
  W8A8_TRY(check_shape(M, 0, K, group_size, 16));
  if (M == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({x, xq}));
  W8A8_TRY(check_ptrs4({scale_a}));
  W8A8_TRY(check_device());
  return launch_row_quant(reinterpret_cast<const __half *>(x), M, K, group_size,
                          127, xq, nullptr, scale_a, as_stream(stream));
}

int w8a8_gemm(const int8_t *xq, const float *scale_a, const int8_t *Wq,
              const float *scale_w, int M, int N, int K, int group_size,
              w8a8_half *y, w8a8_stream_t stream) {
  W8A8_TRY(check_shape(M, N, K, group_size, 16));
  if (M == 0 || N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({xq, Wq, y}));
  W8A8_TRY(check_ptrs4({scale_a, scale_w}));
  W8A8_TRY(check_device());
  return gemm_dispatch(xq, scale_a, Wq, scale_w, M, N, K, group_size, 8,
                       reinterpret_cast<__half *>(y), as_stream(stream));
}

int w8a8_mv(const int8_t *xq, const float *scale_a, const int8_t *Wq,
            const float *scale_w, int M, int N, int K, int group_size,
            w8a8_half *y, w8a8_stream_t stream) {
  if (M != 1) return W8A8_ERR_INVALID_ARG;
  W8A8_TRY(check_shape(M, N, K, group_size, 16));
  if (N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({xq, Wq, y}));
  W8A8_TRY(check_ptrs4({scale_a, scale_w}));
  W8A8_TRY(check_device());
  return launch_gemv_w8a8(xq, scale_a, Wq, scale_w, N, K, group_size,
                          reinterpret_cast<__half *>(y), as_stream(stream));
}

int w4a8_gemm(const int8_t *xq, const float *scale_a, const uint8_t *Wp,
              const float *scale_w, int M, int N, int K, w8a8_half *y,
              w8a8_stream_t stream) {
  W8A8_TRY(check_shape(M, N, K, 0, 32));
  if (M == 0 || N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({xq, Wp, y}));
  W8A8_TRY(check_ptrs4({scale_a, scale_w}));
  W8A8_TRY(check_device());
  return gemm_dispatch(xq, scale_a, Wp, scale_w, M, N, K, 0, 4,
                       reinterpret_cast<__half *>(y), as_stream(stream));
}

int quantize_act_per_token_h(const w8a8_half *x, int M, int K, int group_size,
                             w8a8_half *xq_h, float *scale_a, w8a8_stream_t stream) {
  W8A8_TRY(check_shape(M, 0, K, group_size, 16));
  if (M == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({x, xq_h}));
  W8A8_TRY(check_ptrs4({scale_a}));
  W8A8_TRY(check_device());
  return launch_row_quant_half(reinterpret_cast<const __half *>(x), M, K, group_size,
                               reinterpret_cast<__half *>(xq_h), scale_a, as_stream(stream));
}

int w8a8_gemm_h(const w8a8_half *xq_h, const float *scale_a, const void *Wq,
                const float *scale_w, int M, int N, int K, int group_size, int wbits,
                w8a8_half *y, w8a8_stream_t stream) {
  if (wbits != 8 && wbits != 4) return W8A8_ERR_INVALID_ARG;
  if (wbits == 4 && group_size != 0) return W8A8_ERR_INVALID_ARG;
  W8A8_TRY(check_shape(M, N, K, group_size, wbits == 4 ? 32 : 16));
  if (M == 0 || N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({xq_h, Wq, y}));
  W8A8_TRY(check_ptrs4({scale_a, scale_w}));
  W8A8_TRY(check_device());
  return gemm_h_dispatch(xq_h, scale_a, Wq, scale_w, M, N, K, group_size, wbits,
                         reinterpret_cast<__half *>(y), as_stream(stream));
}

size_t w8a8_linear_workspace_bytes(int M, int K, int group_size) {
  if (M < 0 || K <= 0 || !valid_group_size(K, group_size)) return 0;
  const size_t G = static_cast<size_t>(groups_of(K, group_size));
  const size_t code_bytes = M > 1 ? 2 : 1;  // fp16 codes for the GEMM, int8 for the MV
  return round256(static_cast<size_t>(M) * K * code_bytes) +
         round256(static_cast<size_t>(M) * G * sizeof(float));
}

int linear(const w8a8_half *x, const void *Wq, const float *scale_w, int M,
           int N, int K, int group_size, int wbits, void *workspace,
           size_t ws_bytes, w8a8_half *y, w8a8_stream_t stream) {
  if (wbits != 8 && wbits != 4) return W8A8_ERR_INVALID_ARG;
  if (wbits == 4 && group_size != 0) return W8A8_ERR_INVALID_ARG;
  W8A8_TRY(check_shape(M, N, K, group_size, wbits == 4 ? 32 : 16));
  if (M == 0 || N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({x, Wq, y}));
  W8A8_TRY(check_ptrs4({scale_w}));
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      ws_bytes < w8a8_linear_workspace_bytes(M, K, group_size))
    return W8A8_ERR_WORKSPACE;
  W8A8_TRY(check_device());
  cudaStream_t s = as_stream(stream);
  const size_t code_bytes = M > 1 ? 2 : 1;
  float *sa = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                        round256(static_cast<size_t>(M) * K * code_bytes));
  if (M == 1) {
    // decode: one kernel quantizes the row and streams the weights
    return launch_linear_mv(reinterpret_cast<const __half *>(x), Wq, scale_w, N, K, group_size,
                            wbits, reinterpret_cast<__half *>(y), s);
  }
  if (skinny_supported(M, K, group_size)) {
    // a few rows: one kernel quantizes them and streams the weights (the
    // workspace is checked but not written)
    return launch_linear_rows(reinterpret_cast<const __half *>(x), Wq, scale_w, M, N, K, wbits,
                              reinterpret_cast<__half *>(y), s);
  }
  __half *xq_h = static_cast<__half *>(workspace);
  W8A8_TRY(launch_row_quant_half(reinterpret_cast<const __half *>(x), M, K, group_size, xq_h,
                                 sa, s));
  return gemm_h_dispatch(xq_h, sa, Wq, scale_w, M, N, K, group_size, wbits,
                         reinterpret_cast<__half *>(y), s);
}

int weight_only_gemm(const w8a8_half *x, const void *Wq, const float *scale_w, int M, int N,
                     int K, int group_size, int wbits, w8a8_half *y, w8a8_stream_t stream) {
  if (wbits != 8 && wbits != 4) return W8A8_ERR_INVALID_ARG;
  if (wbits == 4 && group_size != 0) return W8A8_ERR_INVALID_ARG;
  W8A8_TRY(check_shape(M, N, K, group_size, wbits == 4 ? 32 : 16));
  if (M == 0 || N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({x, Wq, y}));
  W8A8_TRY(check_ptrs4({scale_w}));
  W8A8_TRY(check_device());
  return launch_gemm_weight_only(reinterpret_cast<const __half *>(x), Wq, scale_w, M, N, K,
                                 group_size, wbits, reinterpret_cast<__half *>(y),
                                 as_stream(stream));
}

int w8a8_gemm_i32(const int8_t *xq, const void *Wq, int M, int N, int K,
                  int group_size, int wbits, int32_t *acc,
                  w8a8_stream_t stream) {
  if (wbits != 8 && wbits != 4) return W8A8_ERR_INVALID_ARG;
  if (wbits == 4 && group_size != 0) return W8A8_ERR_INVALID_ARG;
  W8A8_TRY(check_shape(M, N, K, group_size, wbits == 4 ? 32 : 16));
  if (M == 0 || N == 0) return W8A8_OK;
  W8A8_TRY(check_ptrs16({xq, Wq, acc}));
  W8A8_TRY(check_device());
  return launch_gemm_tc(xq, false, nullptr, Wq, nullptr, M, N, K, group_size, wbits,
                        nullptr, acc, as_stream(stream));
}

}  // extern "C"
