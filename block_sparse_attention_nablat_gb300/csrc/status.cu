// The library's device status word: kernels record a bounded wait that gave up
// or an out-of-range block index here (first writer wins) instead of trapping.
#include "internal.h"

namespace {
__device__ int g_status;

constexpr int kMaxDevices = 64;
int *g_status_addr[kMaxDevices];
}  // namespace

namespace nabla {

int *device_status_ptr(cudaError_t *err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (!g_status_addr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_status);
    if (*err != cudaSuccess) return nullptr;
    g_status_addr[dev] = static_cast<int *>(p);
  }
  return g_status_addr[dev];
}

}  // namespace nabla
