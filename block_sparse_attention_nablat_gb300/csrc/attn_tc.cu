// K3 -- bf16 block-sparse attention forward (tcgen05 version in progress; the
// CUDA-core kernel serves bf16 until it lands).
#include "internal.h"

namespace nabla {

cudaError_t launch_attn_tc(const void *q, const void *k, const void *v, const Shape &s,
                           const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                           int *status, cudaStream_t st) {
  return launch_attn_simt(q, k, v, NABLA_BF16, s, kv_nb, kv_inds, scale, o, status, st);
}

}  // namespace nabla
