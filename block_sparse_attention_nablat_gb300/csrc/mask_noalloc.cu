// nabla_build_mask_noalloc: the mask builder for callers that cannot allocate
// device memory.  Its scratch (fp32 block means and pooled map) lives in one
// array this file defines in device memory, so the caller passes only inputs
// and outputs.  The array is created when the library's device code is loaded
// and stays reserved on every GPU that loads it until the process exits.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = NABLA_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// Host code must not use this name as an address: on the host it is only a
// stand-in for the symbol.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_mask_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;            // guards the table below: first calls may race
void *g_scratch_addr[kMaxDevices];  // device address of g_mask_scratch, per device

// Set-up, once per device, with that device current.  A cudaDeviceReset
// unloads the library's device code, so an address taken before it is stale;
// the header states that the entry point is then not to be used again on that
// device in this process.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mask_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" nabla_status nabla_build_mask_noalloc(const void *q, const void *k, nabla_dtype dt,
                                                 int B, int S, int h, int D, const uint8_t *sta,
                                                 double thr, int32_t *kv_nb, int32_t *kv_inds,
                                                 nabla_stream_t stream) {
  // host-side checks first: nothing touches the device for a rejected call
  const size_t need = nabla_build_mask_workspace_bytes(B, S, h, D);
  if (need == 0) return NABLA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return NABLA_ERR_UNSUPPORTED;
  if (dt != NABLA_F32 && dt != NABLA_BF16) return NABLA_ERR_INVALID_ARG;
  if (!(thr > 0.0 && thr <= 1.0)) return NABLA_ERR_INVALID_ARG;
  if (!q || !k || !sta || !kv_nb || !kv_inds) return NABLA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return NABLA_ERR_CUDA;
  // The same kernels as nabla_build_mask, with the static array as workspace.
  // Each kernel writes every scratch element it later reads, so the previous
  // call's contents never need clearing.
  return nabla_build_mask(q, k, dt, B, S, h, D, sta, thr, kv_nb, kv_inds, scratch, kScratchBytes,
                          stream);
}
