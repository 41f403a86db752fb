// K4 -- spatio-temporal window (STA) block mask.
//
// FastVideo API reference, page "nabla", NablaAttentionMetadata: the STA mask
// is a block-level [1, 1, S/64, S/64] window shared by all batches and heads,
// precomputed once per run; gist.science NABLA summary, Methodology "Hybrid
// Integration with STA".  The pages do not show how the window is built; the
// reading implemented: on the (T, H, W) block grid, block index (t*H + y)*W + x,
// block j is in row i's window iff |dt| <= wt, |dy| <= wh and |dx| <= ww, with
// no wrap-around.
#include "internal.h"

namespace nabla {
namespace {

__global__ void sta_kernel(int T, int H, int W, int wt, int wh, int ww, uint8_t *sta) {
  const int s1 = T * H * W;
  const long n = (long)s1 * s1;
  for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const int i = (int)(e / s1), j = (int)(e - (long)i * s1);
    const int ti = i / (H * W), yi = (i / W) % H, xi = i % W;
    const int tj = j / (H * W), yj = (j / W) % H, xj = j % W;
    sta[e] = (abs(ti - tj) <= wt && abs(yi - yj) <= wh && abs(xi - xj) <= ww) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_sta(int T, int H, int W, int wt, int wh, int ww, uint8_t *sta,
                       cudaStream_t st) {
  const long n = (long)T * H * W * T * H * W;
  const int blocks = (int)std::min<long>((n + 255) / 256, 4096);
  sta_kernel<<<blocks, 256, 0, st>>>(T, H, W, wt, wh, ww, sta);
  return cudaGetLastError();
}

}  // namespace nabla
