// K7 -- block-sparse attention backward on CUDA cores (fp32 arithmetic).
//
// gist.science NABLA summary, "Dual-Phase Acceleration" and Experimental
// Results: the method trains with the same block mask, so the attention of
// the forward (FastVideo API reference, page "nabla", NablaAttentionImpl.forward)
// is differentiated.  For a query row s with kept tokens J, z = scale q k^T,
// P = softmax(z), o = P v and an upstream gradient dout:
//   dv_u = sum_s P_su dout_s,  dP_su = dout_s . v_u,  delta_s = dout_s . o_s,
//   dz_su = P_su (dP_su - delta_s),  dq_s = scale sum_u dz_su k_u,
//   dk_u = scale sum_s dz_su q_s.
//
// Five kernels:
//   prep     one CTA per query block: delta_s from the stored o, and the row's
//            log-sum-exp over its kept list (base 2, scale folded in), so that
//            P = 2^(z log2(e) - lse2) needs no second normalisation pass;
//   scatter  one warp per query block: sets bit i of key block j's word row
//            for every valid entry j of row i;
//   gather   one warp per key block: lists the query blocks that kept it,
//            ascending (the transposed CSR);
//   dkdv     one CTA per key block: K_j and V_j stay in shared memory while the
//            CTA walks its query blocks, accumulating dK_j and dV_j in registers;
//   dq       one CTA per query block: Q_i and dout_i stay, the CTA walks the
//            kept list and accumulates dQ_i.
// Every 64 x 64 x D product is a register-tiled loop over padded fp32 rows in
// shared memory: thread (tu, tx) of 16 x 16 owns rows tu + 16a and columns
// tx + 16c, so the 16 distinct rows of a warp fall in 16 different banks and
// the other operand is a broadcast.  CSR entries are checked as the forward
// checks them (range, strictly ascending); bad ones are skipped and reported.
#include <cfloat>
#include <type_traits>

#include <cuda_bf16.h>

#include "internal.h"
#include "pdl.cuh"

namespace nabla {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float &d, float x) { d = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 &d, float x) { d = __float2bfloat16_rn(x); }

struct BwdArgs {
  int S, h, s1;
  float scale, scale_log2;
  const int32_t *kv_nb, *kv_inds;
  const float *lse2;          // [B, h, S]: the caller's, or lse2_ws once prep wrote it
  float *lse2_ws, *delta;     // [B, h, S]
  int32_t *qt_nb, *qt_inds;   // [B, h, s1], [B, h, s1, s1]
  uint32_t *bits;             // [B, h, s1, W]
  int words;                  // W = ceil(s1 / 32)
  int *status;
};

// 64 rows of D values (a block of one head) -> fp32 rows of stride D + 1.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float *dst, const T *src, size_t row_stride) {
  for (int e = threadIdx.x; e < 64 * D; e += kThreads) {
    const int r = e / D, d = e - r * D;
    dst[r * (D + 1) + d] = to_f(src[(size_t)r * row_stride + d]);
  }
}

// Validated length of a row's kept list (the forward's rule).
__device__ __forceinline__ int row_count(const BwdArgs &A, size_t row_id) {
  int nb = A.kv_nb[row_id];
  if (nb < 0 || nb > A.s1) {
    if (threadIdx.x == 0) atomicCAS(A.status, kDevOk, kDevBadIndex);
    nb = 0;
  }
  return nb;
}

// Entry n of a kept list is used iff it is in range and above the entry before.
__device__ __forceinline__ bool entry_ok(const int32_t *list, int n, int s1) {
  const int j = list[n];
  return j >= 0 && j < s1 && !(n > 0 && list[n - 1] >= j);
}

// acc[a][c] += sum_d X[tu + 16a][d] * Y[tx + 16c][d] over padded fp32 rows.
template <int D>
__device__ __forceinline__ void tile_dot(const float *X, const float *Y, int tu, int tx,
                                         float (&acc)[4][4]) {
#pragma unroll 4
  for (int d = 0; d < D; ++d) {
    float x[4], y[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) x[a] = X[(tu + 16 * a) * (D + 1) + d];
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = Y[(tx + 16 * c) * (D + 1) + d];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(x[a], y[c], acc[a][c]);
  }
}

// acc[a][c] += sum_r M[r][tu + 16a] * Y[r][tx + 16c]; M is [64][65], Y padded rows.
template <int D>
__device__ __forceinline__ void tile_acc(const float *M, const float *Y, int tu, int tx,
                                         float (&acc)[4][D / 16]) {
#pragma unroll 2
  for (int r = 0; r < 64; ++r) {
    float m[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) m[a] = M[r * 65 + tu + 16 * a];
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const float y = Y[r * (D + 1) + tx + 16 * c];
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[a][c] = fmaf(m[a], y, acc[a][c]);
    }
  }
}

// ---- prep: delta and (kLse) the base-2 log-sum-exp of every query row
template <typename T, int D, bool kLse>
__global__ void __launch_bounds__(kThreads) bwd_prep_kernel(const T *__restrict__ q,
                                                            const T *__restrict__ k,
                                                            const T *__restrict__ o,
                                                            const T *__restrict__ dout,
                                                            BwdArgs A) {
  extern __shared__ float smem[];
  float *Qs = smem;               // [64][D + 1]
  float *Ks = Qs + 64 * (D + 1);  // [64][D + 1]
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x, hh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, tu = tid & 15, tx = tid >> 4;
  const size_t row_stride = (size_t)A.h * D;
  const size_t head_off = (size_t)b * A.S * row_stride + (size_t)hh * D;
  const size_t blk = head_off + (size_t)i * 64 * row_stride;
  const size_t srow = ((size_t)b * A.h + hh) * A.S + (size_t)i * 64;  // [B, h, S] row base

  {  // delta: four threads per row, a quarter of D each
    const int r = tid >> 2, part = tid & 3;
    float a = 0.f;
    const size_t at = blk + (size_t)r * row_stride + part * (D / 4);
#pragma unroll 8
    for (int d = 0; d < D / 4; ++d) a = fmaf(to_f(dout[at + d]), to_f(o[at + d]), a);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    if (part == 0) A.delta[srow + r] = a;
  }
  if (!kLse) return;  // the caller passed the forward's log-sum-exp

  load_rows<T, D>(Qs, q + blk, row_stride);
  const size_t row_id = ((size_t)b * A.h + hh) * A.s1 + i;
  const int nb = row_count(A, row_id);
  const int32_t *list = A.kv_inds + row_id * A.s1;
  float m[4], l[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -FLT_MAX;
    l[a] = 0.f;
  }
  for (int n = 0; n < nb; ++n) {
    if (!entry_ok(list, n, A.s1)) {  // uniform over the CTA
      if (tid == 0) atomicCAS(A.status, kDevOk, kDevBadIndex);
      continue;
    }
    const int j = list[n];
    __syncthreads();  // the previous K block is no longer read
    load_rows<T, D>(Ks, k + head_off + (size_t)j * 64 * row_stride, row_stride);
    __syncthreads();
    // rows tu + 16a of the query block, key columns tx + 16c; a row's 64 columns
    // are spread over the 16 threads tx (eight warps), so the row maximum and
    // sum go through shared memory (K is consumed: its first 1024 floats hold
    // the [16 tx][64 rows] partials)
    float acc[4][4] = {};
    tile_dot<D>(Qs, Ks, tu, tx, acc);
    __syncthreads();
    float *red = Ks;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] *= A.scale_log2;
      red[tx * 64 + tu + 16 * a] =
          fmaxf(fmaxf(acc[a][0], acc[a][1]), fmaxf(acc[a][2], acc[a][3]));
    }
    __syncthreads();
    float mnew[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float mx = m[a];
#pragma unroll 4
      for (int t = 0; t < 16; ++t) mx = fmaxf(mx, red[t * 64 + tu + 16 * a]);
      mnew[a] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) ps += exp2f(acc[a][c] - mnew[a]);
      red[tx * 64 + tu + 16 * a] = ps;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float ps = 0.f;
#pragma unroll 4
      for (int t = 0; t < 16; ++t) ps += red[t * 64 + tu + 16 * a];
      l[a] = l[a] * exp2f(m[a] - mnew[a]) + ps;
      m[a] = mnew[a];
    }
  }
  if (tx == 0) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
      A.lse2_ws[srow + tu + 16 * a] = l[a] > 0.f ? m[a] + log2f(l[a]) : -INFINITY;
  }
}

// ---- scatter: bit i of key block j's word row, for every valid entry of row i
__global__ void __launch_bounds__(kThreads) bwd_scatter_kernel(BwdArgs A, long rows) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long row = (long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int i = (int)(row % A.s1);
  const long bh = row / A.s1;
  int nb = A.kv_nb[row];
  if (nb < 0 || nb > A.s1) {
    if (lane == 0) atomicCAS(A.status, kDevOk, kDevBadIndex);
    nb = 0;
  }
  const int32_t *list = A.kv_inds + (size_t)row * A.s1;
  for (int n = lane; n < nb; n += 32) {
    if (entry_ok(list, n, A.s1)) {
      const int j = list[n];
      atomicOr(&A.bits[((size_t)bh * A.s1 + j) * A.words + (i >> 5)], 1u << (i & 31));
    } else {
      atomicCAS(A.status, kDevOk, kDevBadIndex);
    }
  }
}

// ---- gather: the ascending list of query blocks that kept key block j
__global__ void __launch_bounds__(kThreads) bwd_gather_kernel(BwdArgs A, long rows) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long row = (long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint32_t *w = A.bits + (size_t)row * A.words;
  int32_t *out = A.qt_inds + (size_t)row * A.s1;
  int count = 0;
  for (int w0 = 0; w0 < A.words; w0 += 32) {
    uint32_t word = w0 + lane < A.words ? w[w0 + lane] : 0u;
    const int c = __popc(word);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int at = count + incl - c;
    while (word) {
      const int bit = __ffs(word) - 1;
      out[at++] = (w0 + lane) * 32 + bit;
      word &= word - 1u;
    }
    count += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) A.qt_nb[row] = count;
}

// ---- dK, dV of one key block over the query blocks that kept it
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const T *__restrict__ q,
                                                               const T *__restrict__ k,
                                                               const T *__restrict__ v,
                                                               const T *__restrict__ dout,
                                                               T *__restrict__ dk,
                                                               T *__restrict__ dv, BwdArgs A) {
  constexpr int DC = D / 16;
  extern __shared__ float smem[];
  float *Ks = smem;                 // [64][D + 1]
  float *Vs = Ks + 64 * (D + 1);    // [64][D + 1]
  float *Qs = Vs + 64 * (D + 1);    // [64][D + 1]
  float *dOs = Qs + 64 * (D + 1);   // [64][D + 1]
  float *Ps = dOs + 64 * (D + 1);   // [64 query rows][65]: P[s][u]
  float *dSs = Ps + 64 * 65;        // [64][65]: dz[s][u]
  float *rl = dSs + 64 * 65;        // [64] lse2 of the query rows
  float *rd = rl + 64;              // [64] delta of the query rows
  pdl_launch_dependents();
  pdl_wait();
  const int j = blockIdx.x, hh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, tu = tid & 15, tx = tid >> 4;
  const size_t row_stride = (size_t)A.h * D;
  const size_t head_off = (size_t)b * A.S * row_stride + (size_t)hh * D;
  const size_t bh = (size_t)b * A.h + hh;
  load_rows<T, D>(Ks, k + head_off + (size_t)j * 64 * row_stride, row_stride);
  load_rows<T, D>(Vs, v + head_off + (size_t)j * 64 * row_stride, row_stride);
  float gk[4][DC] = {}, gv[4][DC] = {};
  const int nq = A.qt_nb[bh * A.s1 + j];
  const int32_t *qlist = A.qt_inds + (bh * A.s1 + j) * A.s1;
  for (int n = 0; n < nq; ++n) {
    const int i = qlist[n];
    __syncthreads();  // the previous query block is no longer read
    const size_t blk = head_off + (size_t)i * 64 * row_stride;
    load_rows<T, D>(Qs, q + blk, row_stride);
    load_rows<T, D>(dOs, dout + blk, row_stride);
    if (tid < 64) {
      rl[tid] = A.lse2[bh * A.S + (size_t)i * 64 + tid];
      rd[tid] = A.delta[bh * A.S + (size_t)i * 64 + tid];
    }
    __syncthreads();
    // rows u = tu + 16a of the key block, columns s = tx + 16c of the query block
    float sz[4][4] = {}, dp[4][4] = {};
    tile_dot<D>(Ks, Qs, tu, tx, sz);
    tile_dot<D>(Vs, dOs, tu, tx, dp);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int s = tx + 16 * c;
      const float ls = rl[s], ds = rd[s];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float p = exp2f(fmaf(sz[a][c], A.scale_log2, -ls));
        Ps[s * 65 + tu + 16 * a] = p;
        dSs[s * 65 + tu + 16 * a] = p * (dp[a][c] - ds);
      }
    }
    __syncthreads();
    // dV[u][d] += sum_s P[s][u] dout[s][d];  dK[u][d] += sum_s dz[s][u] q[s][d]
    tile_acc<D>(Ps, dOs, tu, tx, gv);
    tile_acc<D>(dSs, Qs, tu, tx, gk);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const size_t at = head_off + (size_t)(j * 64 + tu + 16 * a) * row_stride;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
      from_f(dk[at + tx + 16 * c], gk[a][c] * A.scale);
      from_f(dv[at + tx + 16 * c], gv[a][c]);
    }
  }
}

// ---- dQ of one query block over its kept list
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const T *__restrict__ q,
                                                             const T *__restrict__ k,
                                                             const T *__restrict__ v,
                                                             const T *__restrict__ dout,
                                                             T *__restrict__ dq, BwdArgs A) {
  constexpr int DC = D / 16;
  extern __shared__ float smem[];
  float *Qs = smem;                 // [64][D + 1]
  float *dOs = Qs + 64 * (D + 1);   // [64][D + 1]
  float *Ks = dOs + 64 * (D + 1);   // [64][D + 1]
  float *Vs = Ks + 64 * (D + 1);    // [64][D + 1]
  float *dSs = Vs + 64 * (D + 1);   // [64 key rows][65]: dz[s][u] stored as [u][s]
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x, hh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, tu = tid & 15, tx = tid >> 4;
  const size_t row_stride = (size_t)A.h * D;
  const size_t head_off = (size_t)b * A.S * row_stride + (size_t)hh * D;
  const size_t bh = (size_t)b * A.h + hh;
  const size_t blk = head_off + (size_t)i * 64 * row_stride;
  load_rows<T, D>(Qs, q + blk, row_stride);
  load_rows<T, D>(dOs, dout + blk, row_stride);
  // rows s = tu + 16a of this query block
  float ls[4], ds[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ls[a] = A.lse2[bh * A.S + (size_t)i * 64 + tu + 16 * a];
    ds[a] = A.delta[bh * A.S + (size_t)i * 64 + tu + 16 * a];
  }
  const size_t row_id = bh * A.s1 + i;
  const int nb = row_count(A, row_id);
  const int32_t *list = A.kv_inds + row_id * A.s1;
  float g[4][DC] = {};
  for (int n = 0; n < nb; ++n) {
    if (!entry_ok(list, n, A.s1)) continue;  // reported by the prep kernel
    const int j = list[n];
    __syncthreads();  // the previous key block is no longer read
    load_rows<T, D>(Ks, k + head_off + (size_t)j * 64 * row_stride, row_stride);
    load_rows<T, D>(Vs, v + head_off + (size_t)j * 64 * row_stride, row_stride);
    __syncthreads();
    float sz[4][4] = {}, dp[4][4] = {};
    tile_dot<D>(Qs, Ks, tu, tx, sz);
    tile_dot<D>(dOs, Vs, tu, tx, dp);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = exp2f(fmaf(sz[a][c], A.scale_log2, -ls[a]));
        dSs[(tx + 16 * c) * 65 + tu + 16 * a] = p * (dp[a][c] - ds[a]);
      }
    __syncthreads();
    // dQ[s][d] += sum_u dz[s][u] k[u][d]
    tile_acc<D>(dSs, Ks, tu, tx, g);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const size_t at = blk + (size_t)(tu + 16 * a) * row_stride;
#pragma unroll
    for (int c = 0; c < DC; ++c) from_f(dq[at + tx + 16 * c], g[a][c] * A.scale);
  }
}

template <int D>
constexpr size_t prep_smem() {
  return sizeof(float) * 2 * 64 * (D + 1);
}
template <int D>
constexpr size_t dkdv_smem() {
  return sizeof(float) * (4 * 64 * (D + 1) + 2 * 64 * 65 + 128);
}
template <int D>
constexpr size_t dq_smem() {
  return sizeof(float) * (4 * 64 * (D + 1) + 64 * 65);
}

template <typename T, int D>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const Shape &s, BwdArgs A, bool have_lse, void *dq,
                         void *dk, void *dv, cudaStream_t st) {
  auto prep = have_lse ? bwd_prep_kernel<T, D, false> : bwd_prep_kernel<T, D, true>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)prep_smem<D>())) != cudaSuccess)
    return e;
  const T *tq = static_cast<const T *>(q), *tk = static_cast<const T *>(k),
          *tv = static_cast<const T *>(v), *to = static_cast<const T *>(o),
          *tdo = static_cast<const T *>(dout);
  const dim3 grid(s.s1, s.h, s.B);
  const long rows = (long)s.B * s.h * s.s1;
  const unsigned warps_grid = (unsigned)((rows + kThreads / 32 - 1) / (kThreads / 32));
  if ((e = launch_pdl(prep, grid, dim3(kThreads), prep_smem<D>(), st, tq, tk, to, tdo, A)) !=
      cudaSuccess)
    return e;
  if ((e = cudaMemsetAsync(A.bits, 0, (size_t)rows * A.words * sizeof(uint32_t), st)) !=
      cudaSuccess)
    return e;
  if ((e = launch_pdl(bwd_scatter_kernel, dim3(warps_grid), dim3(kThreads), 0, st, A, rows)) !=
      cudaSuccess)
    return e;
  if ((e = launch_pdl(bwd_gather_kernel, dim3(warps_grid), dim3(kThreads), 0, st, A, rows)) !=
      cudaSuccess)
    return e;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {  // the products on the tensor cores
    return launch_attn_bwd_tc(q, k, v, dout, s, A.kv_nb, A.kv_inds, A.qt_nb, A.qt_inds, A.lse2,
                              A.delta, A.scale, dq, dk, dv, A.status, st);
  } else {  // fp32: the products on CUDA cores
    auto dkdv = bwd_dkdv_kernel<T, D>;
    auto dqk = bwd_dq_kernel<T, D>;
    if ((e = cudaFuncSetAttribute(dkdv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)dkdv_smem<D>())) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(dqk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)dq_smem<D>())) != cudaSuccess)
      return e;
    if ((e = launch_pdl(dkdv, grid, dim3(kThreads), dkdv_smem<D>(), st, tq, tk, tv, tdo,
                        static_cast<T *>(dk), static_cast<T *>(dv), A)) != cudaSuccess)
      return e;
    return launch_pdl(dqk, grid, dim3(kThreads), dq_smem<D>(), st, tq, tk, tv, tdo,
                      static_cast<T *>(dq), A);
  }
}

}  // namespace

BwdWorkspace bwd_workspace_layout(const Shape &s) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  BwdWorkspace w{};
  const size_t rows = (size_t)s.B * s.h * s.S;
  const size_t blocks = (size_t)s.B * s.h * s.s1;
  w.words = (s.s1 + 31) / 32;
  w.lse2 = 0;
  w.delta = up(rows * 4);
  w.qt_nb = w.delta + up(rows * 4);
  w.qt_inds = w.qt_nb + up(blocks * 4);
  w.bits = w.qt_inds + up(blocks * s.s1 * 4);
  w.o_scratch = w.bits + up(blocks * w.words * 4);
  w.total = w.o_scratch + up((size_t)s.B * s.S * s.h * s.D * 2);
  return w;
}

cudaError_t launch_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dout, nabla_dtype dt, const Shape &s,
                            const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *dq,
                            void *dk, void *dv, void *workspace, int *status, cudaStream_t st) {
  const BwdWorkspace w = bwd_workspace_layout(s);
  char *ws = static_cast<char *>(workspace);
  BwdArgs A{s.S,
            s.h,
            s.s1,
            scale,
            scale * 1.4426950408889634f,
            kv_nb,
            kv_inds,
            lse ? lse : reinterpret_cast<const float *>(ws + w.lse2),
            reinterpret_cast<float *>(ws + w.lse2),
            reinterpret_cast<float *>(ws + w.delta),
            reinterpret_cast<int32_t *>(ws + w.qt_nb),
            reinterpret_cast<int32_t *>(ws + w.qt_inds),
            reinterpret_cast<uint32_t *>(ws + w.bits),
            w.words,
            status};
  if (dt == NABLA_BF16) {
    bool have_lse = lse != nullptr;
    if (!have_lse) {  // the tcgen05 forward gives lse2 (its o goes to scratch)
      const cudaError_t e = launch_attn_tc(q, k, v, s, kv_nb, kv_inds, scale, ws + w.o_scratch,
                                           reinterpret_cast<float *>(ws + w.lse2), status, st);
      if (e != cudaSuccess) return e;
      have_lse = true;
    }
    if (s.D == 64)
      return launch_typed<__nv_bfloat16, 64>(q, k, v, o, dout, s, A, have_lse, dq, dk, dv, st);
    return launch_typed<__nv_bfloat16, 128>(q, k, v, o, dout, s, A, have_lse, dq, dk, dv, st);
  }
  if (s.D == 64) return launch_typed<float, 64>(q, k, v, o, dout, s, A, lse != nullptr, dq, dk, dv, st);
  return launch_typed<float, 128>(q, k, v, o, dout, s, A, lse != nullptr, dq, dk, dv, st);
}

}  // namespace nabla
