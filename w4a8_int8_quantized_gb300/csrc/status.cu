// Device-side error word shared by the kernels that contain bounded waits.
// A kernel whose wait gives up stores a nonzero code (which wait) here and
// returns; w8a8_check_status() reads and clears it.
#include <mutex>

#include "common.cuh"

namespace w8a8 {
namespace {
__device__ unsigned int g_device_error = 0;
}

unsigned int *device_error_word() {
  static unsigned int *cache[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cache[dev] = static_cast<unsigned int *>(p);
  }
  return cache[dev];
}

int read_and_clear_device_error(unsigned int *code) {
  *code = 0;
  if (cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned int)) !=
      cudaSuccess)
    return W8A8_ERR_CUDA;
  if (*code != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int)) !=
        cudaSuccess)
      return W8A8_ERR_CUDA;
  }
  return W8A8_OK;
}

}  // namespace w8a8
