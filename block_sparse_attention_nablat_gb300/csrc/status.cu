// The library's device status word: kernels record a bounded wait that gave up
// or an out-of-range block index here (first writer wins) instead of trapping.
// Also the shared lookup of the driver's tensor-map encoder.
#include "internal.h"
#include "tc_ptx.cuh"

namespace {
__device__ int g_status;

// One CTA waits on an mbarrier that nothing arrives on, through the same
// bounded wait the attention kernel uses; it must give up and record a timeout.
__global__ void bounded_wait_probe(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    nabla::tc::mbar_init(&bar, 1);
    nabla::tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    nabla::tc::mbar_wait(&bar, 0, nullptr, &g_status, nabla::kDevTimeout, limit_ns);
}

}  // namespace

namespace nabla {

// Looked up on every call rather than cached: the lookup is a host-side table
// query, it is safe from any host thread, and it stays right after a
// cudaDeviceReset reloads the library's device code at another address.
int *device_status_ptr(cudaError_t *err) {
  void *p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_status);
  return *err == cudaSuccess ? static_cast<int *>(p) : nullptr;
}

cudaError_t launch_bounded_wait_probe(cudaStream_t st) {
  bounded_wait_probe<<<1, 32, 0, st>>>(20000000ull);  // 20 ms
  return cudaGetLastError();
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(cudaError_t *err) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    *err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                            cudaEnableDefault, &q);
    if (*err != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
      if (*err == cudaSuccess) *err = cudaErrorNotSupported;
      return nullptr;
    }
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *err = cudaSuccess;
  return fn;
}

}  // namespace nabla
