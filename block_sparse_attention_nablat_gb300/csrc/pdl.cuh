// Programmatic dependent launch (PDL) between the kernels of one NABLA step.
//
// Every kernel of the step (pool, pooled map, select, attention) is launched
// with programmatic stream serialization.  At entry it lets the next kernel
// in the stream launch (griddepcontrol.launch_dependents), so that kernel's
// launch and prologue (mbarrier init, TMEM allocation, tensor-map prefetch)
// overlap this kernel's tail.  Before its first global-memory access it waits
// for the previous kernel in the stream to complete and flush its writes
// (griddepcontrol.wait).  The wait is what orders the data.  Everything
// before it touches only shared memory, TMEM and kernel parameters, so a
// kernel of any other origin may precede the call.  Without the launch
// attribute both instructions are no-ops.
//
// The next kernel becomes eligible only once every CTA of this one has
// started or exited, so a dependent CTA that occupies an SM early never keeps
// this kernel's own CTAs from being scheduled.
//
// NABLA_DISABLE_PDL=1 in the environment (read once per process) launches
// with plain stream order instead.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

namespace nabla {

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

inline bool pdl_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("NABLA_DISABLE_PDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

// kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace nabla
