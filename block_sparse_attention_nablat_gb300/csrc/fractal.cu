// Fractal token order: the permutation before (flatten) and after (unflatten)
// the NABLA path.
//
// gist.science NABLA summary, Methodology, "Token Reordering (Fractal
// Flattening)": the tokens of each P x P spatial patch are made contiguous while
// the temporal order is kept; FastVideo API reference, page "nabla": q/k/v reach
// the backend fractal-ordered and nablaT_v2 pools 64-token blocks of that order
// (P = 8: one block = one patch of one frame).  Order used: frames in time order,
// the patches of a frame in raster order, the tokens of a patch row-major.
//
// A token is a contiguous row of h*D elements in both layouts ([B, T, H, W, h, D]
// raster and [B, T*H*W, h, D] fractal), so the permutation moves whole rows: a
// warp per row, 16-byte streaming loads and stores, four in flight per lane.
// HBM-bound: every byte is read once and written once.
#include <cuda_runtime.h>

#include "internal.h"

namespace nabla {
namespace {

constexpr int kThreads = 256;

template <bool kFlatten>
__global__ void __launch_bounds__(kThreads) fractal_kernel(const uint4 *__restrict__ src,
                                                           uint4 *__restrict__ dst, long rows,
                                                           int T, int H, int W, int P,
                                                           int row_vec) {
  const int lane = threadIdx.x & 31;
  const long warps = (long)gridDim.x * (kThreads / 32);
  const long S = (long)T * H * W;
  const int npx = W / P, npy = H / P, pp = P * P;
  for (long f = (long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); f < rows; f += warps) {
    // f: token index in fractal order -> its raster index
    const long b = f / S;
    const long l = f - b * S;
    const long patch = l / pp;
    const int r = (int)(l - patch * pp);
    const int px = (int)(patch % npx);
    const long pr = patch / npx;
    const int py = (int)(pr % npy);
    const long t = pr / npy;
    const int yy = py * P + r / P, xx = px * P + r % P;
    const long raster = b * S + (t * H + yy) * W + xx;
    const uint4 *s = src + (kFlatten ? raster : f) * row_vec;
    uint4 *d = dst + (kFlatten ? f : raster) * row_vec;
    int c = lane;
    for (; c + 96 < row_vec; c += 128) {
      const uint4 v0 = __ldcs(s + c), v1 = __ldcs(s + c + 32), v2 = __ldcs(s + c + 64),
                  v3 = __ldcs(s + c + 96);
      __stcs(d + c, v0);
      __stcs(d + c + 32, v1);
      __stcs(d + c + 64, v2);
      __stcs(d + c + 96, v3);
    }
    for (; c < row_vec; c += 32) __stcs(d + c, __ldcs(s + c));
  }
}

}  // namespace

cudaError_t launch_fractal(const void *src, void *dst, bool flatten, int B, int T, int H, int W,
                           int P, size_t row_bytes, cudaStream_t st) {
  const long rows = (long)B * T * H * W;
  const int row_vec = (int)(row_bytes / 16);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long need = (rows + kThreads / 32 - 1) / (kThreads / 32);
  const long cap = (long)sms * 8;  // 8 resident CTAs of 256 threads per SM
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  if (flatten)
    fractal_kernel<true><<<grid, kThreads, 0, st>>>(static_cast<const uint4 *>(src),
                                                    static_cast<uint4 *>(dst), rows, T, H, W, P,
                                                    row_vec);
  else
    fractal_kernel<false><<<grid, kThreads, 0, st>>>(static_cast<const uint4 *>(src),
                                                     static_cast<uint4 *>(dst), rows, T, H, W, P,
                                                     row_vec);
  return cudaGetLastError();
}

}  // namespace nabla
