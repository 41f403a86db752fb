// K1 -- fused block mean-pool of q and k.
//
// FastVideo API reference, page "nabla", nablaT_v2 "Map estimation": q and k
// are viewed head-major as [B, h, S/64, 64, D] and averaged over the 64 tokens
// of each block; gist.science NABLA summary, Methodology "Downsampling".
//
// Reads q, k in their stored [B, S, h, D] layout (no transpose copy): one CTA
// covers one 64-token block and 64 consecutive 16-byte chunks of the h*D row
// (1 KB of every token row), so every warp load is 512 contiguous bytes. Four
// row groups of 64 threads each sum 16 rows with all 16 loads in flight, then
// the four partial sums are combined in shared memory.  Each mean m is written
// as two tf32 values, hi = m rounded to tf32 and lo = (m - hi) rounded to tf32
// ([B, h, s1, D] each), the operands of the three-term tf32 pooled-map GEMM.
// The q means carry the map's scale log2(e)/sqrt(D) (the map is formed in
// base-2 units), so the GEMM's epilogue stores its accumulators as they are.
// HBM-bound: the algorithmic traffic is the single read of q and k plus the
// (small) means.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "pdl.cuh"

namespace nabla {
namespace {

constexpr int kChunksPerCta = 64;
constexpr int kRowGroups = 4;
constexpr int kRowsPerThread = 64 / kRowGroups;

// q and k are read once: evict-first in L2, so that the stream does not push
// out the pooled map and means that the following kernels read back from L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld_stream(const uint4 *p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

template <typename T>
struct Chunk;

template <>
struct Chunk<float> {
  static constexpr int kElems = 4;
  __device__ static void add(float *acc, const uint4 &u) {
    acc[0] += __uint_as_float(u.x);
    acc[1] += __uint_as_float(u.y);
    acc[2] += __uint_as_float(u.z);
    acc[3] += __uint_as_float(u.w);
  }
};

template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static void add(float *acc, const uint4 &u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[2 * e] += __uint_as_float(w[e] << 16);            // low half = even element
      acc[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);  // high half = odd element
    }
  }
};

__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// grid: (s1, ceil((c1 - c0) / 64), 2 * B); chunks [c0, c1) of the h*D row (the
// heads of one group; C = h*D / elems-per-chunk in all).  z selects (b, q|k).
// qa/ka point at the hi arrays; the lo arrays follow at +lo_off elements.
template <typename T>
__global__ void __launch_bounds__(256) pool_kernel(const T *__restrict__ q,
                                                   const T *__restrict__ k, int S, int h, int D,
                                                   int c0, int c1, float q_scale,
                                                   float *__restrict__ qa,
                                                   float *__restrict__ ka, size_t lo_off) {
  constexpr int E = Chunk<T>::kElems;
  __shared__ float part[kRowGroups][kChunksPerCta * E];
  pdl_launch_dependents();
  pdl_wait();  // q and k are written, and no earlier kernel still reads qa / ka

  const int i = blockIdx.x;
  const int b = blockIdx.z >> 1;
  const bool is_k = blockIdx.z & 1;
  const int s1 = S >> 6;
  const int C = h * D / E;
  const int cx = threadIdx.x % kChunksPerCta;
  const int rg = threadIdx.x / kChunksPerCta;
  const int cb = c0 + blockIdx.y * kChunksPerCta;  // first chunk of this CTA
  const int c = cb + cx;

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  if (c < c1) {
    const uint64_t pol = evict_first_policy();
    const T *src = is_k ? k : q;
    const uint4 *base =
        reinterpret_cast<const uint4 *>(src + ((size_t)b * S + (size_t)i * 64) * h * D) + c;
    uint4 v[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r)
      v[r] = ld_stream(base + (size_t)(rg + kRowGroups * r) * C, pol);
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) Chunk<T>::add(acc, v[r]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) part[rg][cx * E + e] = acc[e];
  __syncthreads();

  // 64 chunks * E elements per CTA, spread over the 256 threads.
  float *dst = is_k ? ka : qa;
  const float mul = is_k ? 1.0f / 64.0f : q_scale * (1.0f / 64.0f);
  for (int e = threadIdx.x; e < kChunksPerCta * E; e += blockDim.x) {
    const int col = cb * E + e;
    if (col >= c1 * E) break;
    const float m = (part[0][e] + part[1][e] + part[2][e] + part[3][e]) * mul;
    const int hh = col / D, d = col - hh * D;
    const size_t at = (((size_t)b * h + hh) * s1 + i) * D + d;
    const float hi = to_tf32(m);
    dst[at] = hi;
    dst[at + lo_off] = to_tf32(m - hi);
  }
}

}  // namespace

cudaError_t launch_pool(const void *q, const void *k, nabla_dtype dt, const Shape &s, int h0,
                        int h1, float *qa, float *ka, size_t lo_off, cudaStream_t st) {
  const int E = dt == NABLA_BF16 ? 8 : 4;  // D is a multiple of 64: heads start on a chunk
  const int c0 = h0 * s.D / E, c1 = h1 * s.D / E;
  const float q_scale = (float)(1.4426950408889634 / sqrt((double)s.D));
  dim3 grid(s.s1, (c1 - c0 + kChunksPerCta - 1) / kChunksPerCta, 2 * s.B);
  if (dt == NABLA_BF16)
    return launch_pdl(pool_kernel<__nv_bfloat16>, grid, dim3(256), 0, st,
                      static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                      s.S, s.h, s.D, c0, c1, q_scale, qa, ka, lo_off);
  return launch_pdl(pool_kernel<float>, grid, dim3(256), 0, st, static_cast<const float *>(q),
                    static_cast<const float *>(k), s.S, s.h, s.D, c0, c1, q_scale, qa, ka,
                    lo_off);
}

}  // namespace nabla
