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
// scale).  One warp per row; the row (s1 <= 2048 values) lives in registers,
// lane l holding the float4 groups at columns 128 m + 4 l .. 128 m + 4 l + 3.
// The softmax is left unnormalised: e_j = 2^(L_j - max), Z = sum e, and the
// running sum of p = e / Z reaches t = 1 - thr exactly where the running sum
// of e reaches t Z, so the cut is taken on e against t Z.  The page sorts the
// row, but the kept set is a suffix of the ascending (e, index) order, so only
// the cut point is needed.  With key(j) = float bits of e_j (monotone, e >= 0):
//   1. one radix pass over the register-resident row: 32 buckets over the key
//      range, each lane adding its blocks' mass into its own column of a
//      [bucket][lane] table; the warp sums the columns, scans the bucket
//      masses and keeps the bucket in which the running sum first reaches t Z;
//   2. the blocks of that bucket (typically a tenth of the row) are copied into
//      a lane-private list in shared memory; further 32-bucket passes run on
//      the list alone until the bucket holds at most 64 blocks;
//   3. those blocks, as 32-bit (key - bucket start, index) pairs, give the
//      exact cut: the first pair (K, i*) in ascending order whose running sum
//      is >= t Z -- by a rank count when they fit one per lane, else by a warp
//      bitonic sort.  A bucket that shrinks to a single key is a run of exact
//      ties, whose running sums base + r e_K give the first kept rank directly.
// Block j is then kept iff key(j) > K, or key(j) == K and j is at or after
// the cut in index order -- the kept set of the sort-based definition,
// evaluated in fp32.  Kept indices, ORed with the STA row, are written in
// ascending order; one packed warp scan gives the offsets of four groups.
#include <cfloat>

#include "internal.h"
#include "pdl.cuh"

namespace nabla {
namespace {

constexpr int kWarps = 4;
constexpr int kBuckets = 32;
constexpr int kSlots = 16;  // lane-private list entries per lane
constexpr int kMaxCand = 64;
constexpr unsigned kAll = 0xffffffffu;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kAll, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kAll, x, o);
  return x;
}
// inclusive prefix sums over the lanes
__device__ __forceinline__ float warp_scan(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kAll, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
__device__ __forceinline__ uint32_t warp_scan_u(uint32_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kAll, x, o);
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
  float mass[kBuckets + 1][32];          // [bucket][lane]: lane-private columns; last row: sink
  uint32_t count[kBuckets / 2 + 1][32];  // 16-bit fields: bucket 2w (low), 2w + 1 (high)
  // [slot][lane]: ((key - list_lo) << 6) | (4 m + e), the entry's key relative to the
  // bucket it was copied from (< 2^26) and its register position; last row: spill
  uint32_t list[kSlots + 1][32];
  uint32_t cand[kMaxCand];
};
constexpr int kMaxRow = 2048;
// after the cut is known the scratch holds the row's kept indices for the store
static_assert(sizeof(WarpScratch) >= kMaxRow * sizeof(int32_t), "row staging fits the scratch");

// The cut range [lo, hi) of keys, the mass below it, and how many blocks it holds.
struct Range {
  uint32_t lo, hi;
  float base;
  int n;
};

// Sum of the lane columns of bucket `lane`: eight 16-byte reads, each quarter
// warp reading eight different 16-byte columns (no bank conflicts).
__device__ __forceinline__ float column_mass(const WarpScratch &ws, int lane) {
  const float4 *row = reinterpret_cast<const float4 *>(ws.mass[lane]);
  float s = 0.f;
#pragma unroll 1
  for (int k0 = 0; k0 < 8; k0 += 4) {  // four loads in flight: the row stays in registers
#pragma unroll
    for (int k = k0; k < k0 + 4; ++k) {
      const float4 v = row[(k + lane) & 7];
      s += (v.x + v.y) + (v.z + v.w);
    }
  }
  return s;
}
__device__ __forceinline__ int column_count(const WarpScratch &ws, int lane) {
  const uint4 *row = reinterpret_cast<const uint4 *>(ws.count[lane >> 1]);
  uint32_t s = 0u;
#pragma unroll 1
  for (int k0 = 0; k0 < 8; k0 += 4) {
#pragma unroll
    for (int k = k0; k < k0 + 4; ++k) {
      const uint4 v = row[(k + (lane >> 1)) & 7];
      s += (v.x + v.y) + (v.z + v.w);
    }
  }
  return (int)((s >> (16 * (lane & 1))) & 0xffffu);
}

// Narrow r to the bucket (of 2^sh keys, bucket 0 starting at d0 << sh) in which
// base + running mass first reaches tz; returns the bucket index.  If fp32
// rounding leaves the sums just short of tz, the cut falls in the last bucket
// with mass (the heaviest block is always kept: the whole row sums to Z > tz).
__device__ __forceinline__ int choose_bucket(Range &r, float bmass, float tz, int sh, uint32_t d0,
                                             int lane) {
  const float cum = warp_scan(bmass, lane);
  const unsigned reach = __ballot_sync(kAll, r.base + cum >= tz);
  const unsigned heavy = __ballot_sync(kAll, bmass > 0.f);
  const int bs = reach   ? __ffs(reach) - 1
                 : heavy ? 31 - __clz(heavy)
                         : (int)(((r.hi - 1u) >> sh) - d0);
  r.base += __shfl_sync(kAll, cum - bmass, bs);
  r.lo = max(r.lo, (d0 + (uint32_t)bs) << sh);
  // the bucket's end can be 2^32 (top-k keys reach the top of the range)
  r.hi = (uint32_t)min((unsigned long long)r.hi, (unsigned long long)(d0 + (uint32_t)bs + 1u) << sh);
  return bs;
}

// Bucket width for a range: 32 buckets of 2^sh keys cover [lo, hi).
__device__ __forceinline__ int bucket_shift(const Range &r) {
  const int top = 31 - __clz(r.lo ^ (r.hi - 1u));
  return top > 4 ? top - 4 : 0;
}

// One 32-bucket pass over the register-resident row (element e of group m is
// column 128 m + 4 lane + e), then the choice of the cut bucket.  RANGED: only
// keys in [r.lo, r.hi) count; the first pass covers every key and needs no
// test.  Excluded elements add into the sink row, so the loop has no branches.
template <int NV, bool FULL, bool RANGED, bool TOPK>
__device__ __forceinline__ void register_pass(WarpScratch &ws, const float (&p)[NV][4], Range &r,
                                              float tz, int lane, int nv, int s1) {
  const int sh = bucket_shift(r);
  const uint32_t d0 = r.lo >> sh, lo = r.lo, w = r.hi - r.lo;
#pragma unroll
  for (int b = 0; b < kBuckets; ++b) ws.mass[b][lane] = 0.f;
#pragma unroll
  for (int m = 0; m < NV; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t u = __float_as_uint(p[m][e]);
      bool in = FULL || (m < nv && 128 * m + 4 * lane + e < s1);
      if (RANGED) in = in && u - lo < w;
      const uint32_t b = in ? (u >> sh) - d0 : (uint32_t)kBuckets;
      ws.mass[b][lane] += TOPK ? 1.0f : p[m][e];  // top-k: every block weighs one
    }
  __syncwarp();
  const float bmass = column_mass(ws, lane);
  __syncwarp();
  choose_bucket(r, bmass, tz, sh, d0, lane);
}

// Copy the blocks with keys in [r.lo, r.hi) into this lane's list and return
// how many there are.  Every element writes slot min(c, kSlots) and only an
// in-range one advances c, so slots [0, c) hold exactly the range's blocks (a
// later block overwrites an out-of-range write); c > kSlots means overflow,
// detected by the caller.  The range spans < 2^26 keys: a bucket of a range of
// keys of e in [0, 1], or a top-k range narrowed to that width first.
template <int NV, bool FULL>
__device__ __forceinline__ int compact_range(WarpScratch &ws, const float (&p)[NV][4],
                                             const Range &r, int lane, int nv, int s1) {
  const uint32_t lo = r.lo, w = r.hi - r.lo;
  int c = 0;
#pragma unroll
  for (int m = 0; m < NV; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t d = __float_as_uint(p[m][e]) - lo;
      const bool in = (FULL || (m < nv && 128 * m + 4 * lane + e < s1)) && d < w;
      ws.list[min(c, kSlots)][lane] = (d << 6) | (uint32_t)(4 * m + e);
      c += in ? 1 : 0;
    }
  return c;
}

// block index of a list entry of this lane
__device__ __forceinline__ uint32_t entry_index(uint32_t word, int lane) {
  return 128u * ((word & 63u) >> 2) + 4u * (uint32_t)lane + (word & 3u);
}

// NV = float4 groups per lane (s1 <= 128 * NV); FULL: s1 == 128 * NV exactly,
// so no column needs a bounds check.
// Rows: grid.y = batch b; the launch covers rows [row0, row0 + nrows) of every
// batch (the heads of one group), a batch being bstride = h * s1 rows apart.
// TOPK: the top-k selector over raw scores (keys = order-preserving bits of the
// score, unit mass per block, cut at count t = n - k + 1, no STA) instead of the
// softmax / cumulative-mass cut.
template <int NV, bool FULL, bool TOPK>
__global__ void __launch_bounds__(kWarps * 32, NV > 12 ? 4 : 5)
    select_kernel(const float *__restrict__ L, long row0, long bstride, int nrows, int s1,
                  const uint8_t *__restrict__ sta, bool sta_words, bool vec_out, float t,
                  int32_t *__restrict__ kv_nb, int32_t *__restrict__ kv_inds) {
  __shared__ __align__(16) WarpScratch scratch[kWarps];  // 16-byte reads and writes
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int local = blockIdx.x * kWarps + warp;
  if (local >= nrows) return;  // uniform per warp
  pdl_wait();  // L is written; no earlier kernel still reads kv_nb / kv_inds
  const long row = blockIdx.y * bstride + row0 + local;
  WarpScratch &ws = scratch[warp];
  const int i = (int)(row % s1);
  const float *Lr = L + row * s1;
  const int nv = FULL ? NV : (s1 + 127) >> 7;
  auto valid = [&](int m, int e) { return FULL || (m < nv && 128 * m + 4 * lane + e < s1); };
  const unsigned lt_mask = (1u << lane) - 1u;

  // STA words of this lane's columns (byte e of word m = column 128 m + 4 lane + e),
  // issued first: consumed only at the end, their latency hides behind the row's work
  const uint8_t *sta_row = sta + (size_t)i * s1;
  uint32_t sw[NV];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int j0 = 128 * m + 4 * lane;
    sw[m] = (!TOPK && sta_words && (FULL || j0 < s1))
                ? *reinterpret_cast<const uint32_t *>(sta_row + j0)
                : 0u;
  }
  // ---- load the row; column of element e of group m is 128 m + 4 lane + e
  float p[NV][4];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int j0 = 128 * m + 4 * lane;
    if (FULL || (m < nv && (s1 & 3) == 0 && j0 + 3 < s1)) {
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
  float tz;
  uint32_t kmin, kmax;
  if constexpr (TOPK) {
    // order-preserving key of a float (sign-magnitude -> unsigned); the largest
    // pattern is held back so that kmax + 1 does not wrap
    uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int m = 0; m < NV; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t x = __float_as_uint(p[m][e]);
        if ((x << 1) == 0u) x = 0u;  // -0 ranks with +0 (they tie)
        uint32_t u = min(x ^ ((x >> 31) ? 0xffffffffu : 0x80000000u), 0xfffffffeu);
        if (!valid(m, e)) u = 0u;
        else {
          kmn = min(kmn, u);
          kmx = max(kmx, u);
        }
        p[m][e] = __uint_as_float(u);
      }
    tz = t;
    kmin = __reduce_min_sync(kAll, kmn);
    kmax = __reduce_max_sync(kAll, kmx);
  } else {
    // ---- unnormalised softmax e = 2^(L - max) (fp32); Z = sum e
    float mx = -FLT_MAX;
  #pragma unroll
    for (int m = 0; m < NV; ++m)
      mx = fmaxf(mx, fmaxf(fmaxf(p[m][0], p[m][1]), fmaxf(p[m][2], p[m][3])));
    mx = warp_max(mx);
    float z0 = 0.f, z1 = 0.f, emin = FLT_MAX, emax = 0.f;
  #pragma unroll
    for (int m = 0; m < NV; ++m)
  #pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (valid(m, e)) {
          // fmaxf maps a NaN (from non-finite logits) to 0: every key then lies in
          // [kmin, kmax], which bounds the bucket indices of the first pass
          p[m][e] = fmaxf(exp2_approx(p[m][e] - mx), 0.f);
          emin = fminf(emin, p[m][e]);
          emax = fmaxf(emax, p[m][e]);
        } else {
          p[m][e] = 0.f;
        }
        if (e & 1)
          z1 += p[m][e];
        else
          z0 += p[m][e];
      }
    tz = t * warp_sum(z0 + z1);
    // e >= 0, so float order is the order of the bits
    kmin = __reduce_min_sync(kAll, __float_as_uint(emin));
    kmax = __reduce_max_sync(kAll, __float_as_uint(emax));
  }
  // ---- cut: kept iff key > K, or key == K and tie rank (index order) >= R
  const bool keep_all = !(t > 0.f);
  uint32_t K = 0u;
  int R = 0;
  int ties_at_K = 2;  // > 1 unless the cut key is known to be unique
  if (!keep_all) {
    Range r{kmin, kmax + 1u, 0.f, s1};
    bool done = false;
    // a bucket of one key is a run of exact ties: running sums base + (r + 1) e_K
    // at tie ranks r = 0 .. n - 1
    auto finish_ties = [&](const Range &rr) {
      const float ek = TOPK ? 1.0f : __uint_as_float(rr.lo);
      K = rr.lo;
      R = ek > 0.f ? min(max(0, (int)ceilf((tz - rr.base) / ek) - 1), rr.n - 1) : 0;
      ties_at_K = rr.n;
      done = true;
    };
    int c = 0;  // this lane's list entries (more than kSlots: overflow)
    uint32_t list_lo = 0u;  // key offset of the list entries
    if (r.hi - r.lo == 1u) {
      finish_ties(r);
    } else {
      register_pass<NV, FULL, false, TOPK>(ws, p, r, tz, lane, nv, s1);
      // top-k keys span up to 2^32: narrow until the range packs into a list entry
#pragma unroll 1
      while (TOPK && !done && r.hi - r.lo > (1u << 26)) {
        if (r.hi - r.lo == 1u)
          finish_ties(r);
        else
          register_pass<NV, FULL, true, TOPK>(ws, p, r, tz, lane, nv, s1);
      }
      c = compact_range<NV, FULL>(ws, p, r, lane, nv, s1);
      list_lo = r.lo;
      r.n = (int)__reduce_add_sync(kAll, (unsigned)c);
      // rare: the cut bucket overflows a lane's list; narrow it in registers
#pragma unroll 1
      for (int level = 1; !done && (int)__reduce_max_sync(kAll, (unsigned)c) > kSlots; ++level) {
        if (r.hi - r.lo == 1u) {
          finish_ties(r);
        } else if (level == 7) {  // unreachable: each pass takes 5 bits off a < 2^30 range
          K = r.lo;
          R = 0;
          done = true;
        } else {
          register_pass<NV, FULL, true, TOPK>(ws, p, r, tz, lane, nv, s1);
          c = compact_range<NV, FULL>(ws, p, r, lane, nv, s1);
          list_lo = r.lo;
          r.n = (int)__reduce_add_sync(kAll, (unsigned)c);
        }
      }
    }
    // -- passes over the list
    const int nl = min(c, kSlots);
    const int cmax = (int)__reduce_max_sync(kAll, (unsigned)nl);
#pragma unroll 1
    for (int pass = 0; pass < 8 && !done; ++pass) {
      if (r.n <= kMaxCand && r.hi - r.lo <= (1u << 21)) {
        // ---- exact finish: (key - lo) packs with an 11-bit block index
        const uint32_t lo = r.lo, w = r.hi - r.lo;
        int nc = 0;
#pragma unroll 1
        for (int sl = 0; sl < cmax; ++sl) {
          const uint32_t word = ws.list[sl][lane];
          const uint32_t key = list_lo + (word >> 6);
          const bool in = sl < nl && key - lo < w;
          const unsigned bal = __ballot_sync(kAll, in);
          const int at = nc + __popc(bal & lt_mask);
          if (in && at < kMaxCand) ws.cand[at] = ((key - lo) << 11) | entry_index(word, lane);
          nc += __popc(bal);
        }
        nc = min(nc, kMaxCand);
        __syncwarp();
        if (nc <= 32) {
          // rank count: running sum at a pair = base + mass of the pairs below it
          const uint32_t my = lane < nc ? ws.cand[lane] : kAll;
          const float ev = lane < nc ? (TOPK ? 1.0f : __uint_as_float((my >> 11) + lo)) : 0.f;
          float below = 0.f;
#pragma unroll 4
          for (int sl = 0; sl < nc; ++sl) {
            const uint32_t o = __shfl_sync(kAll, my, sl);
            const float eo = __shfl_sync(kAll, ev, sl);
            if (o < my) below += eo;
          }
          const bool reach = lane < nc && r.base + below + ev >= tz;
          uint32_t cut = __reduce_min_sync(kAll, reach ? my : kAll);
          if (cut == kAll) cut = __reduce_max_sync(kAll, lane < nc ? my : 0u);  // keep the heaviest
          const uint32_t kd = cut >> 11;
          K = kd + lo;
          R = __popc(__ballot_sync(kAll, lane < nc && (my >> 11) == kd && my < cut));
          ties_at_K = __popc(__ballot_sync(kAll, lane < nc && (my >> 11) == kd));
        } else {
          // ascending bitonic sort of 64 keys held two per lane (positions lane, lane + 32)
          uint32_t a = ws.cand[lane];
          uint32_t b = lane + 32 < nc ? ws.cand[lane + 32] : kAll;
#pragma unroll
          for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
              if (j == 32) {  // partners are the two values of one lane; k == 64 ascends
                const uint32_t x = min(a, b), y = max(a, b);
                a = x;
                b = y;
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  uint32_t &x = h ? b : a;
                  const int pos = lane + 32 * h;
                  const uint32_t y = __shfl_xor_sync(kAll, x, j);
                  const bool take_min = ((pos & j) == 0) == ((pos & k) == 0);
                  x = take_min ? min(x, y) : max(x, y);
                }
              }
            }
          }
          const float pa = TOPK ? 1.0f : __uint_as_float((a >> 11) + lo);  // nc > 32: real
          const float pb = lane + 32 < nc ? (TOPK ? 1.0f : __uint_as_float((b >> 11) + lo)) : 0.f;
          const float ca = warp_scan(pa, lane);
          const float cb = warp_scan(pb, lane) + __shfl_sync(kAll, ca, 31);
          const unsigned ba = __ballot_sync(kAll, r.base + ca >= tz);
          const unsigned bb = __ballot_sync(kAll, lane + 32 < nc && r.base + cb >= tz);
          const int q = ba ? __ffs(ba) - 1 : bb ? 32 + __ffs(bb) - 1 : nc - 1;
          const uint32_t cut = q < 32 ? __shfl_sync(kAll, a, q & 31) : __shfl_sync(kAll, b, q & 31);
          const uint32_t kd = cut >> 11;
          K = kd + lo;
          R = __popc(__ballot_sync(kAll, lane < q && (a >> 11) == kd)) +
              __popc(__ballot_sync(kAll, lane + 32 < q && (b >> 11) == kd));
          ties_at_K = __popc(__ballot_sync(kAll, (a >> 11) == kd)) +
                      __popc(__ballot_sync(kAll, lane + 32 < nc && (b >> 11) == kd));
        }
        done = true;
        break;
      }
      if (r.hi - r.lo == 1u) {
        finish_ties(r);
        break;
      }
      const int sh = bucket_shift(r);
      const uint32_t d0 = r.lo >> sh, lo = r.lo, w = r.hi - r.lo;
#pragma unroll
      for (int b = 0; b < kBuckets; ++b) ws.mass[b][lane] = 0.f;
#pragma unroll
      for (int b = 0; b < kBuckets / 2; ++b) ws.count[b][lane] = 0u;
#pragma unroll 1
      for (int sl = 0; sl < cmax; ++sl) {
        const uint32_t key = list_lo + (ws.list[sl][lane] >> 6);
        const bool in = sl < nl && key - lo < w;
        const uint32_t b = in ? (key >> sh) - d0 : (uint32_t)kBuckets;  // else the sink
        ws.mass[b][lane] += TOPK ? 1.0f : __uint_as_float(key);
        ws.count[b >> 1][lane] += 1u << (16 * (b & 1u));
      }
      __syncwarp();
      const float bmass = column_mass(ws, lane);
      const int bcount = column_count(ws, lane);
      __syncwarp();
      const int bs = choose_bucket(r, bmass, tz, sh, d0, lane);
      r.n = __shfl_sync(kAll, bcount, bs);
    }
    if (!done) {  // unreachable: a < 2^25 key range narrows to one key in 5 list passes
      K = r.lo;
      R = 0;
    }
  }

  // ---- keep flags: one nibble per group, bit e = column 128 m + 4 lane + e
  uint32_t kn[NV];
  const bool ranked = !keep_all && ties_at_K > 1;  // ties at the cut: rank them (rare)
  auto sta_nibble = [&](int m) -> uint32_t {
    if (TOPK) return 0u;
    const int j0 = 128 * m + 4 * lane;
    uint32_t x = sw[m];  // STA flags of the four columns, byte e = column j0 + e
    if (!sta_words) {
      x = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j0 + e < s1) x |= (uint32_t)sta_row[j0 + e] << (8 * e);
    }
    // nonzero bytes -> bits 0, 8, 16, 24 -> nibble bits 0..3 (the multiply's
    // partial products land on distinct bits, so nothing carries)
    x |= x >> 4;
    x |= x >> 2;
    x |= x >> 1;
    return ((x & 0x01010101u) * 0x00204081u >> 21) & 0xfu;
  };
  auto valid_nibble = [&](int m) -> uint32_t {
    uint32_t v = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) v |= (uint32_t)valid(m, e) << e;
    return v;
  };
  if (!ranked) {
    const uint32_t Kc = keep_all ? 0u : K;  // keep_all: every key qualifies
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      uint32_t keep = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) keep |= (uint32_t)(__float_as_uint(p[m][e]) >= Kc) << e;
      kn[m] = (keep | sta_nibble(m)) & valid_nibble(m);
    }
  } else {
    int ties = 0;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      uint32_t tie = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (valid(m, e) && __float_as_uint(p[m][e]) == K) tie |= 1u << e;
      const uint32_t tc = (uint32_t)__popc(tie);
      const uint32_t tincl = warp_scan_u(tc, lane);
      int rank = ties + (int)(tincl - tc);
      ties += (int)__shfl_sync(kAll, tincl, 31);
      uint32_t keep = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t u = __float_as_uint(p[m][e]);
        if (u > K || (u == K && valid(m, e) && rank++ >= R)) keep |= 1u << e;
      }
      kn[m] = (keep | sta_nibble(m)) & valid_nibble(m);
    }
  }
  // ---- emit kept indices in ascending order: byte k of the packed scan is
  // group m0 + k (a group holds at most 128 kept blocks: no carries).  They are
  // staged in the warp's scratch (free now) and then stored row-contiguously.
  int32_t *stage = reinterpret_cast<int32_t *>(&ws);
  __syncwarp();  // every lane is done with the scratch's histogram / list contents
  int count = 0;
#pragma unroll
  for (int m0 = 0; m0 < NV; m0 += 4) {
    uint32_t wcount = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (m0 + k < NV) wcount |= (uint32_t)__popc(kn[m0 + k]) << (8 * k);
    const uint32_t incl = warp_scan_u(wcount, lane);
    const uint32_t total = __shfl_sync(kAll, incl, 31);
    const uint32_t excl = incl - wcount;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int m = m0 + k;
      if (m >= NV) break;
      int at = count + (int)((excl >> (8 * k)) & 0xffu);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kn[m] & (1u << e)) stage[at++] = 128 * m + 4 * lane + e;
      count += (int)((total >> (8 * k)) & 0xffu);
    }
  }
  __syncwarp();
  int32_t *out = kv_inds + row * s1;
  if (vec_out) {  // rows start 16-byte aligned: four indices per lane per store
    int i = 4 * lane;
    for (; i + 4 <= count; i += 128)
      *reinterpret_cast<int4 *>(out + i) = *reinterpret_cast<const int4 *>(stage + i);
    for (; i < count; ++i) out[i] = stage[i];  // this lane's part of the tail
  } else {
    for (int i = lane; i < count; i += 32) out[i] = stage[i];
  }
  if (lane == 0) kv_nb[row] = count;
}

struct SelectLaunch {
  dim3 grid;
  cudaStream_t st;
  const float *L;
  long row0, bstride;
  int nrows, s1;
  const uint8_t *sta;
  float t;
  int32_t *kv_nb, *kv_inds;
};

template <int NV, bool TOPK>
cudaError_t launch_nv(const SelectLaunch &a) {
  const bool words = (a.s1 & 3) == 0 && (reinterpret_cast<uintptr_t>(a.sta) & 3u) == 0;
  const bool vec = (a.s1 & 3) == 0 && (reinterpret_cast<uintptr_t>(a.kv_inds) & 15u) == 0;
  auto kern = a.s1 == 128 * NV ? select_kernel<NV, true, TOPK> : select_kernel<NV, false, TOPK>;
  return launch_pdl(kern, a.grid, dim3(kWarps * 32), 0, a.st, a.L, a.row0, a.bstride, a.nrows,
                    a.s1, a.sta, words, vec, a.t, a.kv_nb, a.kv_inds);
}

}  // namespace

namespace {

template <bool TOPK>
cudaError_t select_dispatch(const float *L, const Shape &s, int h0, int h1, const uint8_t *sta,
                            float t, int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st) {
  const int nrows = (h1 - h0) * s.s1;
  SelectLaunch a{dim3((unsigned)((nrows + kWarps - 1) / kWarps), (unsigned)s.B),
                 st,
                 L,
                 (long)h0 * s.s1,
                 (long)s.h * s.s1,
                 nrows,
                 s.s1,
                 sta,
                 t,
                 kv_nb,
                 kv_inds};
  const int nv = (s.s1 + 127) / 128;
  if (nv <= 1) return launch_nv<1, TOPK>(a);
  if (nv <= 2) return launch_nv<2, TOPK>(a);
  if (nv <= 4) return launch_nv<4, TOPK>(a);
  if (nv <= 8) return launch_nv<8, TOPK>(a);
  if (nv <= 12) return launch_nv<12, TOPK>(a);
  return launch_nv<16, TOPK>(a);
}

}  // namespace

cudaError_t launch_select(const float *L, const Shape &s, int h0, int h1, const uint8_t *sta,
                          float t, int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st) {
  return select_dispatch<false>(L, s, h0, h1, sta, t, kv_nb, kv_inds, st);
}

cudaError_t launch_select_topk(const float *L, const Shape &s, int h0, int h1, int topk,
                               int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st) {
  // unit mass per block: the running count reaches s1 - topk + 1 at the first
  // kept block; topk = s1 keeps every block (t = 0)
  const float t = topk >= s.s1 ? 0.f : (float)(s.s1 - topk + 1);
  return select_dispatch<true>(L, s, h0, h1, nullptr, t, kv_nb, kv_inds, st);
}

}  // namespace nabla
