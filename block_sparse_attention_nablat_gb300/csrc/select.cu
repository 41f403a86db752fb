// K2b -- row softmax, ascending running-sum cut, STA union and CSR emit.
//
// FastVideo API reference, page "nabla", nablaT_v2: softmax over each row of
// the pooled map, "Map binarization" (sort ascending, running sum, keep
// entries whose running sum is >= 1 - thr, flags back in block order), logical
// OR with the STA window, then kv_nb = row count and kv_inds = kept blocks
// first.  gist.science NABLA summary, Methodology "CDF Thresholding" and
// "Hybrid Integration with STA".
//
// The pooled map arrives in base-2 units (L * log2 e, folded into the map's
// scale), so p = 2^(L - max) / sum.  One warp per row; the row (s1 <= 2048
// values) lives in registers, lane l holding the float4 groups at columns
// 128 m + 4 l .. 128 m + 4 l + 3.  The page sorts the row, but the kept set is
// a suffix of the ascending (p, index) order, so only the cut point is needed.
// With key(j) = float bits of p_j (monotone since p >= 0):
//   1. radix passes over the key range: 32 buckets per pass, each lane adding
//      its blocks' mass and count into its own column of a [bucket][lane]
//      shared-memory table (no atomics, no bank conflicts); the warp sums the
//      columns, scans the 32 bucket masses and keeps the bucket in which the
//      running sum first reaches t = 1 - thr;
//   2. as soon as that bucket holds at most 64 blocks, they are compacted into
//      shared memory as 32-bit (key - bucket start, index) pairs, sorted by a
//      warp bitonic network and scanned from the mass below the bucket, which
//      gives the exact cut: the first pair (K, i*) whose running sum is >= t;
//   3. a bucket that shrinks to a single key is a run of exact ties: their
//      running sums are base + r * p, so the first kept rank follows directly.
// Block j is then kept iff key(j) > K, or key(j) == K and j is at or after
// the cut in index order -- the kept set of the sort-based definition,
// evaluated in fp32.  Kept indices, ORed with the STA row, are written in
// ascending order: per 128-column group, four warp ballots give every lane its
// output position by population counts.
#include <cfloat>

#include "internal.h"

namespace nabla {
namespace {

constexpr int kWarps = 8;
constexpr int kBuckets = 32;
constexpr int kMaxCand = 64;

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
// inclusive prefix sums over the lanes
__device__ __forceinline__ float warp_scan(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
__device__ __forceinline__ int warp_scan_i(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct WarpScratch {
  float mass[kBuckets][33];       // [bucket][lane] (+1 pad): lane-private columns
  uint32_t count[kBuckets / 4][33];  // byte b & 3 of word [b >> 2][lane]: a lane holds <= 64 blocks
  uint32_t cand[kMaxCand];   // ((key - bucket start) << 11) | index
};

// Ascending bitonic sort of 64 32-bit keys held two per lane (positions lane, lane+32).
__device__ __forceinline__ void warp_sort64(uint32_t &a, uint32_t &b, int lane) {
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // partners are the two values of one lane; k == 64 ascends everywhere
        const uint32_t lo = min(a, b), hi = max(a, b);
        a = lo;
        b = hi;
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t &x = h ? b : a;
          const int pos = lane + 32 * h;
          const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
          // the lower position of a pair keeps the smaller key in an ascending run
          const bool take_min = ((pos & j) == 0) == ((pos & k) == 0);
          x = take_min ? min(x, y) : max(x, y);
        }
      }
    }
  }
}

// NV = float4 groups per lane (s1 <= 128 * NV); FULL: s1 == 128 * NV exactly,
// so no column needs a bounds check.
template <int NV, bool FULL>
__global__ void __launch_bounds__(kWarps * 32) select_kernel(const float *__restrict__ L,
                                                             long rows, int s1,
                                                             const uint8_t *__restrict__ sta,
                                                             bool sta_words, float t,
                                                             int32_t *__restrict__ kv_nb,
                                                             int32_t *__restrict__ kv_inds) {
  __shared__ WarpScratch scratch[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long row = (long)blockIdx.x * kWarps + warp;
  if (row >= rows) return;  // uniform per warp
  WarpScratch &ws = scratch[warp];
  const int i = (int)(row % s1);
  const float *Lr = L + row * s1;
  const int nv = FULL ? NV : (s1 + 127) >> 7;
  const bool vec = FULL || (s1 & 3) == 0;
  auto valid = [&](int m, int e) { return FULL || (m < nv && 128 * m + 4 * lane + e < s1); };

  // ---- load the row; column of element e of group m is 128 m + 4 lane + e
  float p[NV][4];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int j0 = 128 * m + 4 * lane;
    if (FULL || (m < nv && vec && j0 + 3 < s1)) {
      const float4 v = *reinterpret_cast<const float4 *>(Lr + j0);
      p[m][0] = v.x;
      p[m][1] = v.y;
      p[m][2] = v.z;
      p[m][3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) p[m][e] = valid(m, e) ? Lr[j0 + e] : -FLT_MAX;
    }
  }
  // ---- softmax (fp32, base 2)
  float mx = -FLT_MAX;
#pragma unroll
  for (int m = 0; m < NV; ++m)
    mx = fmaxf(mx, fmaxf(fmaxf(p[m][0], p[m][1]), fmaxf(p[m][2], p[m][3])));
  mx = warp_max(mx);
  float z0 = 0.f, z1 = 0.f;
#pragma unroll
  for (int m = 0; m < NV; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[m][e] = valid(m, e) ? exp2_approx(p[m][e] - mx) : 0.f;
      if (e & 1)
        z1 += p[m][e];
      else
        z0 += p[m][e];
    }
  const float inv_z = 1.0f / warp_sum(z0 + z1);
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int m = 0; m < NV; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[m][e] *= inv_z;
      if (valid(m, e)) {
        const uint32_t u = __float_as_uint(p[m][e]);
        kmin = min(kmin, u);
        kmax = max(kmax, u);
      }
    }
  kmin = warp_umin(kmin);
  kmax = warp_umax(kmax);

  // ---- cut: kept iff key > K, or key == K and tie rank (index order) >= R
  uint32_t K = 0u;
  int R = 0;
  int ties_at_K = 2;  // > 1 unless the cut key is known to be unique
  if (t > 0.f) {
    uint32_t lo = kmin, hi = kmax + 1u;
    float base = 0.f;  // mass of keys below lo
    int in_range = s1;  // blocks with key in [lo, hi)
    // each pass takes 5 bits off a range of < 2^30 keys: 7 passes always suffice
    for (int pass = 0; pass < 7; ++pass) {
      if (hi - lo == 1u) {  // a single key: a run of exact ties
        // running sums base + (r + 1) pk at tie ranks r = 0 .. in_range - 1
        const float pk = __uint_as_float(lo);
        K = lo;
        R = pk > 0.f ? min(max(0, (int)ceilf((t - base) / pk) - 1), in_range - 1) : 0;
        ties_at_K = in_range;
        break;
      }
      const int top = 31 - __clz(lo ^ (hi - 1u));
      const int sh = top > 4 ? top - 4 : 0;
      const uint32_t d0 = lo >> sh;
#pragma unroll
      for (int b = 0; b < kBuckets; ++b) ws.mass[b][lane] = 0.f;
#pragma unroll
      for (int b = 0; b < kBuckets / 4; ++b) ws.count[b][lane] = 0u;
#pragma unroll
      for (int m = 0; m < NV; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t u = __float_as_uint(p[m][e]);
          if (valid(m, e) && u >= lo && u < hi) {
            const int b = (int)((u >> sh) - d0);
            ws.mass[b][lane] += p[m][e];
            ws.count[b >> 2][lane] += 1u << (8 * (b & 3));
          }
        }
      __syncwarp();
      // lane b sums bucket b over the lanes (fixed order: deterministic)
      float bmass = 0.f;
      int bcount = 0;
      const int cshift = 8 * (lane & 3);
#pragma unroll
      for (int l = 0; l < 32; ++l) {
        bmass += ws.mass[lane][l];
        bcount += (int)((ws.count[lane >> 2][l] >> cshift) & 0xffu);
      }
      __syncwarp();
      const float cum = warp_scan(bmass, lane);
      const unsigned bal = __ballot_sync(0xffffffffu, base + cum >= t);
      // The whole row sums to 1 > t; if fp32 rounding leaves the bucket sums just
      // short of t, the cut falls in the last bucket of the range (the heaviest
      // block is always kept).
      const int bs = bal ? __ffs(bal) - 1 : (int)(((hi - 1u) >> sh) - d0);
      base += __shfl_sync(0xffffffffu, cum - bmass, bs);
      const int cnt = __shfl_sync(0xffffffffu, bcount, bs);
      in_range = cnt;
      lo = max(lo, (d0 + (uint32_t)bs) << sh);
      hi = min(hi, (d0 + (uint32_t)bs + 1u) << sh);
      const int wbits = 32 - __clz(hi - lo - 1u);  // bits spanned by the new range
      if (cnt <= kMaxCand && wbits <= 21) {
        // ---- exact finish on the bucket's blocks: (key - lo) packs with an
        // 11-bit block index into 32 bits
        int nc = 0;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          uint32_t flags = 0u;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t u = __float_as_uint(p[m][e]);
            if (valid(m, e) && u >= lo && u < hi) flags |= 1u << e;
          }
          const int c = __popc(flags);
          const int incl_c = warp_scan_i(c, lane);
          int at = nc + incl_c - c;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (flags & (1u << e))
              ws.cand[at++] = ((__float_as_uint(p[m][e]) - lo) << 11) | (uint32_t)(128 * m + 4 * lane + e);
          nc += __shfl_sync(0xffffffffu, incl_c, 31);
        }
        __syncwarp();
        uint32_t a = lane < nc ? ws.cand[lane] : 0xffffffffu;
        uint32_t b = lane + 32 < nc ? ws.cand[lane + 32] : 0xffffffffu;
        __syncwarp();
        warp_sort64(a, b, lane);
        // running sums in sorted order: positions lane (a) and lane + 32 (b)
        const float pa = lane < nc ? __uint_as_float((a >> 11) + lo) : 0.f;
        const float pb = lane + 32 < nc ? __uint_as_float((b >> 11) + lo) : 0.f;
        const float ca = warp_scan(pa, lane);
        const float cb = warp_scan(pb, lane) + __shfl_sync(0xffffffffu, ca, 31);
        const unsigned ba = __ballot_sync(0xffffffffu, lane < nc && base + ca >= t);
        const unsigned bb = __ballot_sync(0xffffffffu, lane + 32 < nc && base + cb >= t);
        int q;  // sorted position of the cut
        if (ba)
          q = __ffs(ba) - 1;
        else if (bb)
          q = 32 + __ffs(bb) - 1;
        else
          q = nc - 1;  // rounding: keep the heaviest candidate
        const uint32_t cut =
            q < 32 ? __shfl_sync(0xffffffffu, a, q & 31) : __shfl_sync(0xffffffffu, b, q & 31);
        const uint32_t kd = cut >> 11;
        K = kd + lo;
        // tie rank of the cut among blocks with key K = sorted candidates before it with key K
        const bool ta = lane < q && (a >> 11) == kd;
        const bool tb = lane + 32 < q && (b >> 11) == kd;
        R = __popc(__ballot_sync(0xffffffffu, ta)) + __popc(__ballot_sync(0xffffffffu, tb));
        const bool ea = lane < nc && (a >> 11) == kd, eb = lane + 32 < nc && (b >> 11) == kd;
        ties_at_K = __popc(__ballot_sync(0xffffffffu, ea)) + __popc(__ballot_sync(0xffffffffu, eb));
        break;
      }
      if (pass == 6) {  // unreachable for keys of p in (0, 1]; keep a defined result
        K = lo;
        R = 0;
      }
    }
  }

  // ---- emit kept indices in ascending order
  const uint8_t *sta_row = sta + (size_t)i * s1;
  int32_t *out = kv_inds + row * s1;
  const bool keep_all = !(t > 0.f);
  const unsigned lt_mask = (1u << lane) - 1u;
  int count = 0, ties = 0;
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    if (!FULL && m >= nv) break;
    const int j0 = 128 * m + 4 * lane;
    uint32_t sbits;  // STA flags of the four columns, byte e = column j0 + e
    if (sta_words) {  // s1 % 4 == 0 and a 4-byte aligned STA: one word per lane
      sbits = (FULL || j0 < s1) ? *reinterpret_cast<const uint32_t *>(sta_row + j0) : 0u;
    } else {
      sbits = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j0 + e < s1) sbits |= (uint32_t)sta_row[j0 + e] << (8 * e);
    }
    int rank = 0;
    if (ties_at_K > 1 && !keep_all) {  // rank blocks with key K in index order
      uint32_t tie = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (valid(m, e) && __float_as_uint(p[m][e]) == K) tie |= 1u << e;
      const int tc = __popc(tie);
      const int tincl = warp_scan_i(tc, lane);
      rank = ties + tincl - tc;
      ties += __shfl_sync(0xffffffffu, tincl, 31);
    }
    uint32_t keep = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!valid(m, e)) continue;
      const uint32_t u = __float_as_uint(p[m][e]);
      bool k;
      if (keep_all)
        k = true;
      else if (u != K)
        k = u > K;
      else
        k = rank++ >= R;
      if (k || ((sbits >> (8 * e)) & 0xffu) != 0u) keep |= 1u << e;
    }
    const unsigned b0 = __ballot_sync(0xffffffffu, keep & 1u);
    const unsigned b1 = __ballot_sync(0xffffffffu, keep & 2u);
    const unsigned b2 = __ballot_sync(0xffffffffu, keep & 4u);
    const unsigned b3 = __ballot_sync(0xffffffffu, keep & 8u);
    int at = count + __popc(b0 & lt_mask) + __popc(b1 & lt_mask) + __popc(b2 & lt_mask) +
             __popc(b3 & lt_mask);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (keep & (1u << e)) out[at++] = j0 + e;
    count += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
  }
  if (lane == 0) kv_nb[row] = count;
}

template <int NV>
void launch_nv(unsigned grid, cudaStream_t st, const float *L, long rows, int s1,
               const uint8_t *sta, float t, int32_t *kv_nb, int32_t *kv_inds) {
  const bool words = (s1 & 3) == 0 && (reinterpret_cast<uintptr_t>(sta) & 3u) == 0;
  if (s1 == 128 * NV)
    select_kernel<NV, true>
        <<<grid, kWarps * 32, 0, st>>>(L, rows, s1, sta, words, t, kv_nb, kv_inds);
  else
    select_kernel<NV, false>
        <<<grid, kWarps * 32, 0, st>>>(L, rows, s1, sta, words, t, kv_nb, kv_inds);
}

}  // namespace

cudaError_t launch_select(const float *L, const Shape &s, const uint8_t *sta, float t,
                          int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st) {
  const long rows = (long)s.B * s.h * s.s1;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  const int nv = (s.s1 + 127) / 128;
  if (nv <= 1)
    launch_nv<1>(grid, st, L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (nv <= 2)
    launch_nv<2>(grid, st, L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (nv <= 4)
    launch_nv<4>(grid, st, L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (nv <= 8)
    launch_nv<8>(grid, st, L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else if (nv <= 12)
    launch_nv<12>(grid, st, L, rows, s.s1, sta, t, kv_nb, kv_inds);
  else
    launch_nv<16>(grid, st, L, rows, s.s1, sta, t, kv_nb, kv_inds);
  return cudaGetLastError();
}

}  // namespace nabla
