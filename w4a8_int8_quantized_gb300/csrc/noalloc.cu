// linear() for callers that cannot allocate device memory.
//
// linear() needs a workspace for the quantized activations (the INT8 codes
// -- stored as fp16 values when M > 1 -- and their fp32 scales), which the
// caller allocates.  Some callers have no allocator to hand on their
// execution path: a serving runtime's per-request path where cudaMalloc is
// forbidden because it can synchronize the device and fail under memory
// pressure, or a plugin running inside a host framework that owns all
// device memory through its own pool and gives plugins no allocation hook.
// linear_noalloc() serves them: its workspace is a fixed array in this
// library's device memory (kScratchBytes, 8 MiB), so it allocates nothing.
//
// Costs and rules of that array:
//  * every GPU that loads the library holds the 8 MiB until the process
//    exits;
//  * all calls on a device share it: two calls whose kernels overlap on the
//    GPU (different streams without ordering between them) race on it and
//    give wrong results.  Calls on one stream are ordered and safe;
//  * it keeps the last call's contents.  Nothing in it needs to start at
//    zero: each call writes every code and scale it later reads;
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, once per device, with that device current);
//    make that first call before any stream capture begins.
#include <mutex>

#include "common.cuh"

namespace w8a8 {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;

// In host code this name is only a stand-in for the symbol, not a device
// address: the address the kernels get comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_linear_scratch[kScratchBytes];

// Device address of g_linear_scratch on the current device, looked up once
// per device.  nullptr if the lookup fails.
void *scratch_address() {
  static void *addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_linear_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace w8a8

extern "C" int linear_noalloc(const w8a8_half *x, const void *Wq, const float *scale_w, int M,
                              int N, int K, int group_size, int wbits, w8a8_half *y,
                              w8a8_stream_t stream) {
  if (wbits != 8 && wbits != 4) return W8A8_ERR_INVALID_ARG;
  if (wbits == 4 && group_size != 0) return W8A8_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K <= 0 || K > w8a8::kMaxK) return W8A8_ERR_INVALID_ARG;
  if (!w8a8::valid_group_size(K, group_size)) return W8A8_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return W8A8_OK;
  const size_t need = w8a8_linear_workspace_bytes(M, K, group_size);
  if (need == 0) return W8A8_ERR_INVALID_ARG;
  if (need > w8a8::kScratchBytes) return W8A8_ERR_WORKSPACE;  // does not fit the fixed array
  const int dev_status = w8a8::check_device();
  if (dev_status != W8A8_OK) return dev_status;
  void *ws = w8a8::scratch_address();
  if (ws == nullptr) return W8A8_ERR_CUDA;
  return linear(x, Wq, scale_w, M, N, K, group_size, wbits, ws, w8a8::kScratchBytes, y, stream);
}
