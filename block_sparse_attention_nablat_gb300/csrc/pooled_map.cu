// K2a -- pooled map L = qa ka^T / sqrt(D) per (batch, head), fp32.
//
// FastVideo API reference, page "nabla", nablaT_v2 "Map estimation": the block
// means are multiplied (qa @ ka^T) and the result divided by sqrt(D) before the
// row softmax; gist.science NABLA summary, Methodology "Reduced Attention".
//
// CUDA-core fp32 GEMM: 128x128 output tile per CTA, k-slab of 16, 256 threads
// each owning an 8x8 register tile (two 4-row by two 4-column float4 strips so
// that the shared-memory reads are conflict-free float4 loads), double-buffered
// shared tiles.  fp32 keeps the logits within ~1e-6 of the exact value, which
// the ascending running-sum cut needs (an order swap of two near-equal blocks
// at the cut would change both of their running sums by a whole block mass).
#include "internal.h"

namespace nabla {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, PAD = 4;

// grid: (ceil(s1/128), ceil(s1/128), B*h)
__global__ void __launch_bounds__(256, 2) pooled_map_kernel(const float *__restrict__ qa,
                                                            const float *__restrict__ ka, int s1,
                                                            int D, float scale,
                                                            float *__restrict__ L) {
  __shared__ __align__(16) float As[2][BK][BM + PAD];
  __shared__ __align__(16) float Bs[2][BK][BN + PAD];

  const size_t bh = blockIdx.z;
  const float *A = qa + bh * s1 * D;
  const float *Bm = ka + bh * s1 * D;
  float *C = L + bh * (size_t)s1 * s1;
  const int row0 = blockIdx.y * BM, col0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;

  // global -> register staging: 128 rows x 16 k = 512 float4 per operand, 2 per thread
  float4 ra[2], rb[2];
  auto load = [&](int k0) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = tid + 256 * u;
      const int r = idx >> 2, kq = (idx & 3) * 4;
      const int gr = row0 + r, gc = col0 + r;
      ra[u] = gr < s1 ? *reinterpret_cast<const float4 *>(A + (size_t)gr * D + k0 + kq)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      rb[u] = gc < s1 ? *reinterpret_cast<const float4 *>(Bm + (size_t)gc * D + k0 + kq)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = tid + 256 * u;
      const int r = idx >> 2, kq = (idx & 3) * 4;
      As[buf][kq + 0][r] = ra[u].x;
      As[buf][kq + 1][r] = ra[u].y;
      As[buf][kq + 2][r] = ra[u].z;
      As[buf][kq + 3][r] = ra[u].w;
      Bs[buf][kq + 0][r] = rb[u].x;
      Bs[buf][kq + 1][r] = rb[u].y;
      Bs[buf][kq + 2][r] = rb[u].z;
      Bs[buf][kq + 3][r] = rb[u].w;
    }
  };

  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[a][c] = 0.f;

  const int nk = D / BK;
  load(0);
  store(0);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load((kt + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
    }
    if (kt + 1 < nk) {
      store(buf ^ 1);
      __syncthreads();
    }
  }

#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const int r = row0 + (x < 4 ? ty * 4 + x : 64 + ty * 4 + (x - 4));
    if (r >= s1) continue;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = col0 + half * 64 + tx * 4;
      float4 o = make_float4(acc[x][half * 4 + 0] * scale, acc[x][half * 4 + 1] * scale,
                             acc[x][half * 4 + 2] * scale, acc[x][half * 4 + 3] * scale);
      if (c + 3 < s1 && (s1 & 3) == 0) {
        *reinterpret_cast<float4 *>(C + (size_t)r * s1 + c) = o;
      } else {
        const float ov[4] = {o.x, o.y, o.z, o.w};
        for (int e = 0; e < 4; ++e)
          if (c + e < s1) C[(size_t)r * s1 + c + e] = ov[e];
      }
    }
  }
}

}  // namespace

cudaError_t launch_pooled_map(const float *qa, const float *ka, const Shape &s, float *L,
                              cudaStream_t st) {
  const int nt = (s.s1 + BM - 1) / BM;
  dim3 grid(nt, nt, s.B * s.h);
  const float scale = (float)(1.0 / sqrt((double)s.D));
  pooled_map_kernel<<<grid, 256, 0, st>>>(qa, ka, s.s1, s.D, scale, L);
  return cudaGetLastError();
}

}  // namespace nabla
