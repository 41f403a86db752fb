// K2b -- row softmax, ascending running-sum cut, STA union and CSR emit.
//
// FastVideo API reference, page "nabla", nablaT_v2: softmax over each row of
// the pooled map, "Map binarization" (sort ascending, running sum, keep
// entries whose running sum is >= 1 - thr, flags back in block order), logical
// OR with the STA window, then kv_nb = row count and kv_inds = kept blocks
// first.  gist.science NABLA summary, Methodology "CDF Thresholding" and
// "Hybrid Integration with STA".
//
// One warp per row; the row (s1 <= 2048 values) lives in registers, lane l
// holding blocks l, l+32, ...  The page sorts the row, but the kept set is a
// suffix of the ascending order, so only the cut point is needed: with
// key(j) = float bits of p_j (monotone, p >= 0) and ties ordered by block
// index, block j is kept iff its running sum c(j) >= t.  The cut key is found
// by a most-significant-digit radix select over the key range: each pass
// splits the current range into 32 buckets, sums the probability mass per
// bucket (one shared-memory histogram column per lane, conflict-free), and a
// warp scan finds the bucket in which the running sum first reaches t.  After
// the range shrinks to one key, ties at that key are resolved in block-index
// order.  The result is exactly the kept set of the sort-based definition,
// evaluated in fp32.  Kept indices are then compacted in ascending order with
// warp ballots, ORed with the STA row, and written with coalesced stores.
#include <cfloat>

#include "internal.h"

namespace nabla {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ uint32_t warp_umin(uint32_t x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = min(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ uint32_t warp_umax(uint32_t x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// MAXM = register slots per lane (s1 <= 32 * MAXM); M = ceil(s1 / 32) at run time.
template <int MAXM>
__global__ void __launch_bounds__(kWarps * 32) select_kernel(const float *__restrict__ L,
                                                             long rows, int s1,
                                                             const uint8_t *__restrict__ sta,
                                                             float t, int32_t *__restrict__ kv_nb,
                                                             int32_t *__restrict__ kv_inds) {
  __shared__ float hist_all[kWarps][32][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long row = (long)blockIdx.x * kWarps + warp;
  if (row >= rows) return;  // uniform per warp
  float(*hist)[33] = hist_all[warp];
  const int i = (int)(row % s1);
  const float *Lr = L + row * s1;
  const int M = (s1 + 31) >> 5;

  // softmax of the row (fp32)
  float p[MAXM];
  float mx = -FLT_MAX;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    const int j = m * 32 + lane;
    p[m] = (m < M && j < s1) ? Lr[j] : -FLT_MAX;
    mx = fmaxf(mx, p[m]);
  }
  mx = warp_max(mx);
  float z = 0.f;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    const int j = m * 32 + lane;
    const float e = (m < M && j < s1) ? expf(p[m] - mx) : 0.f;
    p[m] = e;
    z += e;
  }
  z = warp_sum(z);
  const float inv_z = 1.0f / z;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    const int j = m * 32 + lane;
    p[m] *= inv_z;
    if (m < M && j < s1) {
      const uint32_t u = __float_as_uint(p[m]);
      kmin = min(kmin, u);
      kmax = max(kmax, u);
    }
  }
  kmin = warp_umin(kmin);
  kmax = warp_umax(kmax);

  // radix select of the cut key: smallest key K with F(K) = sum_{key <= K} p >= t.
  uint32_t lo = kmin, hi = kmax + 1u;
  float base = 0.f;  // mass of keys < lo
  bool none = false;  // running sum never reaches t: the CDF part keeps nothing
  const bool keep_all = !(t > 0.f);
  bool first = true;
  // each pass shrinks the range by >= 16x; keys of p in (0, 1] span < 2^30, so 8 passes suffice
  for (int pass = 0; pass < 8 && !keep_all && hi - lo > 1u; ++pass) {
    const int top = 31 - __clz(lo ^ (hi - 1u));
    const int sh = top > 4 ? top - 4 : 0;
    const uint32_t d0 = lo >> sh;
#pragma unroll
    for (int b = 0; b < 32; ++b) hist[b][lane] = 0.f;
    __syncwarp();
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      const int j = m * 32 + lane;
      const uint32_t u = __float_as_uint(p[m]);
      if (m < M && j < s1 && u >= lo && u < hi) hist[(u >> sh) - d0][lane] += p[m];
    }
    __syncwarp();
    float mass = 0.f;
#pragma unroll
    for (int l = 0; l < 32; ++l) mass += hist[lane][l];
    float cum = mass;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, cum, o);
      if (lane >= o) cum += y;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, base + cum >= t);
    int bs;
    if (bal == 0u) {
      if (first) {
        none = true;
        break;
      }
      // fp32 rounding of the sub-bucket sums fell just short of t: take the last
      // bucket that intersects the range
      bs = (int)(((hi - 1u) >> sh) - d0);
    } else {
      bs = __ffs(bal) - 1;
    }
    base += __shfl_sync(0xffffffffu, cum - mass, bs);
    const uint32_t nlo = (d0 + (uint32_t)bs) << sh;
    const uint32_t nhi = (d0 + (uint32_t)bs + 1u) << sh;
    lo = max(lo, nlo);
    hi = min(hi, nhi);
    first = false;
    __syncwarp();
  }

  // emit: kept = key > K, or key == K and (tie rank) running sum >= t, or STA.
  const uint8_t *sta_row = sta + (size_t)i * s1;
  int32_t *out = kv_inds + row * s1;
  const float pk = __uint_as_float(lo);
  const unsigned lt_mask = (1u << lane) - 1u;
  int count = 0, ties = 0;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    if (m >= M) break;
    const int j = m * 32 + lane;
    const bool valid = j < s1;
    const uint32_t u = __float_as_uint(p[m]);
    const bool tie = valid && !keep_all && !none && u == lo;
    const unsigned tb = __ballot_sync(0xffffffffu, tie);
    const int rank = ties + __popc(tb & (lt_mask | (1u << lane)));
    ties += __popc(tb);
    bool cdf;
    if (keep_all)
      cdf = valid;
    else
      cdf = valid && !none && (u > lo || (tie && base + (float)rank * pk >= t));
    const bool keep = valid && (cdf || sta_row[j] != 0);
    const unsigned kb = __ballot_sync(0xffffffffu, keep);
    if (keep) out[count + __popc(kb & lt_mask)] = j;
    count += __popc(kb);
  }
  if (lane == 0) kv_nb[row] = count;
}

}  // namespace

cudaError_t launch_select(const float *L, const Shape &s, const uint8_t *sta, float t,
                          int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st) {
  const long rows = (long)s.B * s.h * s.s1;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  const int M = (s.s1 + 31) / 32;
  if (M <= 4)
    select_kernel<4><<<grid, kWarps * 32, 0, st>>>(L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (M <= 16)
    select_kernel<16><<<grid, kWarps * 32, 0, st>>>(L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (M <= 32)
    select_kernel<32><<<grid, kWarps * 32, 0, st>>>(L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (M <= 48)
    select_kernel<48><<<grid, kWarps * 32, 0, st>>>(L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else
    select_kernel<64><<<grid, kWarps * 32, 0, st>>>(L, rows, s.s1, sta, t, kv_nb, kv_inds);
  return cudaGetLastError();
}

}  // namespace nabla
