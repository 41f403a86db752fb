// K3f -- block-sparse attention forward on CUDA cores (fp32 storage).
//
// FastVideo API reference, page "nabla", NablaAttentionImpl.forward: attention
// over the block mask of full 64x64 blocks, non-causal, default scale;
// gist.science NABLA summary, Methodology "Expansion".  tcgen05 has no fp32
// MMA and tf32 would not hold fp32 accuracy, so fp32 inputs run here in fp32.
//
// One CTA per (query block, head, batch), 256 threads: thread (r, part) owns
// query row r and a quarter of the kept block's 64 key columns for QK^T and a
// quarter of the D output columns for PV.  Online softmax (running max and sum
// per row, base-2 exponent with the scale folded in); the four threads of a
// row are adjacent lanes and combine their partial max/sum with shuffles.
#include <cfloat>

#include <cuda_bf16.h>

#include "internal.h"
#include "pdl.cuh"

namespace nabla {
namespace {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float &d, float x) { d = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 &d, float x) { d = __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_simt_kernel(const T *__restrict__ q,
                                                        const T *__restrict__ k,
                                                        const T *__restrict__ v, int S, int h,
                                                        const int32_t *__restrict__ kv_nb,
                                                        const int32_t *__restrict__ kv_inds,
                                                        float scale_log2, T *__restrict__ o,
                                                        float *__restrict__ lse, int *status) {
  constexpr int DQ = D / 4;
  extern __shared__ float smem[];
  float *Qs = smem;               // [64][D + 1]
  float *Ks = Qs + 64 * (D + 1);  // [64][D + 1]
  float *Vs = Ks + 64 * (D + 1);  // [64][D]
  float *Ps = Vs + 64 * D;        // [64][65]

  const int i = blockIdx.x, hh = blockIdx.y, b = blockIdx.z;
  const int s1 = S >> 6;
  const int tid = threadIdx.x, r = tid >> 2, part = tid & 3;
  const size_t row_stride = (size_t)h * D;
  const size_t head_off = (size_t)b * S * row_stride + (size_t)hh * D;
  pdl_launch_dependents();
  pdl_wait();  // kv_nb / kv_inds and q, k, v are written; no earlier kernel still reads o

  for (int e = tid; e < 64 * D; e += 256) {
    const int rr = e / D, d = e - rr * D;
    Qs[rr * (D + 1) + d] = to_f(q[head_off + (size_t)(i * 64 + rr) * row_stride + d]);
  }

  const size_t row_id = ((size_t)b * h + hh) * s1 + i;
  int nb = kv_nb[row_id];
  if (nb < 0 || nb > s1) {
    if (tid == 0) atomicCAS(status, kDevOk, kDevBadIndex);
    nb = 0;
  }
  const int32_t *list = kv_inds + row_id * s1;

  float m_run = -FLT_MAX, l_run = 0.f;
  float acc[DQ];
#pragma unroll
  for (int e = 0; e < DQ; ++e) acc[e] = 0.f;

  for (int n = 0; n < nb; ++n) {
    const int j = list[n];
    if (j < 0 || j >= s1 || (n > 0 && list[n - 1] >= j)) {  // uniform over the CTA
      if (tid == 0) atomicCAS(status, kDevOk, kDevBadIndex);
      continue;
    }
    __syncthreads();  // previous block's K/V/P no longer read
    for (int e = tid; e < 64 * D; e += 256) {
      const int rr = e / D, d = e - rr * D;
      const size_t g = head_off + (size_t)(j * 64 + rr) * row_stride + d;
      Ks[rr * (D + 1) + d] = to_f(k[g]);
      Vs[rr * D + d] = to_f(v[g]);
    }
    __syncthreads();

    float s[16];
    float mx = -FLT_MAX;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float *kr = Ks + (part * 16 + c) * (D + 1);
      const float *qr = Qs + r * (D + 1);
      float a = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) a = fmaf(qr[d], kr[d], a);
      s[c] = a * scale_log2;
      mx = fmaxf(mx, s[c]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float alpha = exp2f(m_run - m_new);
    float ps = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float pv = exp2f(s[c] - m_new);
      Ps[r * 65 + part * 16 + c] = pv;
      ps += pv;
    }
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    l_run = l_run * alpha + ps;
    m_run = m_new;
#pragma unroll
    for (int e = 0; e < DQ; ++e) acc[e] *= alpha;
    __syncwarp();  // the row's four P quarters come from lanes of this warp
    for (int c = 0; c < 64; ++c) {
      const float pc = Ps[r * 65 + c];
      const float *vr = Vs + c * D + part * DQ;
#pragma unroll
      for (int e = 0; e < DQ; ++e) acc[e] = fmaf(pc, vr[e], acc[e]);
    }
  }

  const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
  if (lse && part == 0)  // base-2 log-sum-exp of the row's scaled scores
    lse[((size_t)b * h + hh) * S + (size_t)i * 64 + r] =
        l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
  T *orow = o + head_off + (size_t)(i * 64 + r) * row_stride + part * DQ;
#pragma unroll
  for (int e = 0; e < DQ; ++e) from_f(orow[e], acc[e] * inv);
}

template <typename T, int D>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const Shape &s,
                         const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                         float *lse, int *status, cudaStream_t st) {
  const size_t smem = sizeof(float) * (64 * (D + 1) * 2 + 64 * D + 64 * 65);
  auto kern = attn_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(s.s1, s.h, s.B);
  return launch_pdl(kern, grid, dim3(256), smem, st, static_cast<const T *>(q),
                    static_cast<const T *>(k), static_cast<const T *>(v), s.S, s.h, kv_nb, kv_inds,
                    scale * 1.4426950408889634f, static_cast<T *>(o), lse, status);
}

}  // namespace

cudaError_t launch_attn_simt(const void *q, const void *k, const void *v, nabla_dtype dt,
                             const Shape &s, const int32_t *kv_nb, const int32_t *kv_inds,
                             float scale, void *o, float *lse, int *status, cudaStream_t st) {
  if (dt == NABLA_F32)
    return s.D == 64
               ? launch_typed<float, 64>(q, k, v, s, kv_nb, kv_inds, scale, o, lse, status, st)
               : launch_typed<float, 128>(q, k, v, s, kv_nb, kv_inds, scale, o, lse, status, st);
  return s.D == 64 ? launch_typed<__nv_bfloat16, 64>(q, k, v, s, kv_nb, kv_inds, scale, o, lse,
                                                      status, st)
                   : launch_typed<__nv_bfloat16, 128>(q, k, v, s, kv_nb, kv_inds, scale, o, lse,
                                                       status, st);
}

}  // namespace nabla
