// Helpers shared by the tcgen05 attention kernels (forward and backward):
// the pair-of-blocks work units with their entry bitmaps, packed fp32 pair
// arithmetic, mbarrier ring positions, the in-kernel choice of the pairing
// stride, and the TMA map of a [B, S, h, D] bf16 tensor.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "internal.h"

namespace nabla {
namespace tcattn {

constexpr int kMaxWords = 64;  // s1 <= 2048 blocks -> 64 bitmap words

struct UnitInfo {
  uint32_t a[kMaxWords];  // kept by the first query block of the pair
  uint32_t b[kMaxWords];  // kept by the second
  int n;                  // union size
  int start;              // first key block of the walk (the walk wraps around)
};

struct Cursor {
  int w;
  uint32_t m;
};

constexpr int kMaxEntries = 32 * kMaxWords;  // entries of a unit (s1 <= 2048)

// Warp-wide: the unit's entry count, and each entry's two membership bits
// (bit 0: first block of the pair, bit 1: second) written to fl[0 .. n) in
// walk order: ascending key block from block `start`, then around from block 0
// (start = 0: plain ascending order).  Lane l lists the entries of bitmap words
// 2l and 2l + 1, starting where the lanes before it end.  Lets the threads
// that walk a unit's entries read one byte per entry instead of each
// scanning the bitmaps.
__device__ __forceinline__ int list_entries(const UnitInfo &inf, uint8_t *fl, int lane,
                                            int start = 0) {
  static_assert(kMaxWords == 64, "two bitmap words per lane");
  const uint32_t u0 = inf.a[2 * lane] | inf.b[2 * lane];
  const uint32_t u1 = inf.a[2 * lane + 1] | inf.b[2 * lane + 1];
  const int mine = __popc(u0) + __popc(u1);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int pos = incl - mine;
  const int n = __shfl_sync(0xffffffffu, incl, 31);
  // entries below `start` go last: r0 of them, so entry e is walked at (e - r0) mod n
  const int w0 = start >> 5;
  auto below = [&](int w, uint32_t u) -> int {
    return w < w0 ? __popc(u) : w == w0 ? __popc(u & ((1u << (start & 31)) - 1u)) : 0;
  };
  const int r0 = __reduce_add_sync(0xffffffffu, (unsigned)(below(2 * lane, u0) +
                                                           below(2 * lane + 1, u1)));
#pragma unroll
  for (int hw = 0; hw < 2; ++hw) {
    const int w = 2 * lane + hw;
    const uint32_t aw = inf.a[w], bw = inf.b[w];
    for (uint32_t m = hw ? u1 : u0; m; m &= m - 1u) {
      const int bit = __ffs(m) - 1;
      const int at = pos >= r0 ? pos - r0 : pos - r0 + n;
      fl[at] = (uint8_t)(((aw >> bit) & 1u) | (((bw >> bit) & 1u) << 1));
      ++pos;
    }
  }
  return n;
}

// A cursor over the unit's entries that starts at key block `start` and wraps
// around: the walk order list_entries writes for the same start.
__device__ __forceinline__ Cursor cursor_at(const UnitInfo &inf, int start) {
  const int w0 = start >> 5;
  return Cursor{w0, (inf.a[w0] | inf.b[w0]) & (~0u << (start & 31))};
}
// Next entry of a cursor_at walk; called at most n times per unit.
__device__ __forceinline__ int next_entry_wrap(const UnitInfo &inf, Cursor &c, int start) {
  const int w0 = start >> 5;
  for (int i = 0; c.m == 0u && i <= kMaxWords; ++i) {
    c.w = c.w + 1 == kMaxWords ? 0 : c.w + 1;
    c.m = inf.a[c.w] | inf.b[c.w];
    if (c.w == w0) c.m &= (1u << (start & 31)) - 1u;  // back at the start word
  }
  const int bit = c.m ? __ffs(c.m) - 1 : 0;
  c.m &= c.m - 1u;
  return c.w * 32 + bit;
}

__device__ __forceinline__ int next_entry(const UnitInfo &inf, Cursor &c, uint32_t &flags) {
  while (c.m == 0u && c.w + 1 < kMaxWords) {
    ++c.w;
    c.m = inf.a[c.w] | inf.b[c.w];
  }
  const int bit = c.m ? __ffs(c.m) - 1 : 0;
  c.m &= c.m - 1u;
  flags = ((inf.a[c.w] >> bit) & 1u) | (((inf.b[c.w] >> bit) & 1u) << 1);
  return c.w * 32 + bit;
}

// Query block `side` (0 or 1) of pair pr at stride d: pairs run through groups
// of 2d consecutive blocks, (g 2d + o, g 2d + o + d) for o < d.
__device__ __forceinline__ int pair_block(int pr, int side, int d) {
  const int g = pr / d;
  return 2 * g * d + (pr - g * d) + side * d;
}

struct Unit {
  int b, hh, pr;
};
__device__ __forceinline__ Unit decode(long u, int npairs, int h) {
  const long bh = u / npairs;
  Unit r;
  r.pr = (int)(u - bh * npairs);
  r.b = (int)(bh / h);
  r.hh = (int)(bh - (long)r.b * h);
  return r;
}

// packed fp32 pairs (sm_100+ f32x2 arithmetic)
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Ring position: slot index and phase parity advanced without division.
template <int N>
struct Ring {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == (uint32_t)N) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Pairing stride: the candidate d (1, or any d with 2d dividing s1) whose
// pairs have the smallest total list union over a fixed sample of pairs.  Run
// by all threads of every CTA (the first 12 warps do the counting) on scratch shared memory
// before the roles start; integer counts make the choice identical in every
// CTA.  L: any struct with B, S, h and the CSR lists kv_nb, kv_inds.  With
// mean_union given, the sample is counted even when d = 1 is the only
// candidate, and *mean_union receives the chosen d's mean union size (>= 1).
constexpr int kMaxCands = 24, kSamples = 16;
struct StrideScratch {
  uint32_t bits[12][kMaxWords];
  unsigned long long total[kMaxCands];
  int cand[kMaxCands];
  int ncand, chosen, mean_union;
};

template <class L>
__device__ int choose_pair_stride(const L &P, StrideScratch *sc, int *mean_union = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  if (threadIdx.x == 0) {
    int n = 0;
    sc->cand[n++] = 1;
    for (int d = 2; 2 * d <= s1 && n < kMaxCands; ++d)
      if (s1 % (2 * d) == 0) sc->cand[n++] = d;
    sc->ncand = n;
    for (int c = 0; c < kMaxCands; ++c) sc->total[c] = 0ull;
  }
  __syncthreads();
  const int ncand = sc->ncand;
  if (ncand > 1 || mean_union) {
    // at most 12 warps take part (one scratch row each); the others skip to the barrier
    const int nw = (int)(blockDim.x >> 5) < 12 ? (int)(blockDim.x >> 5) : 12;
    uint32_t *bits = sc->bits[warp < 12 ? warp : 0];
    for (int t = warp; warp < nw && t < ncand * kSamples; t += nw) {
      const int c = t / kSamples, k = t - c * kSamples;
      const int d = sc->cand[c];
      // the same units for every candidate, spread over all heads and rows
      const long u = (long)(((unsigned long long)k * 2654435761ull) % (unsigned long long)units);
      const Unit un = decode(u, npairs, P.h);
      const long bh = (long)un.b * P.h + un.hh;
      int cnt[2];
      const int32_t *list[2];
#pragma unroll
      for (int side = 0; side < 2; ++side) {
        const int qb = pair_block(un.pr, side, d);
        const size_t row = (size_t)bh * s1 + (qb < s1 ? qb : 0);
        const int n = qb < s1 ? P.kv_nb[row] : 0;
        cnt[side] = n < 0 ? 0 : (n > s1 ? s1 : n);
        list[side] = P.kv_inds + row * s1;
      }
      for (int w = lane; w < kMaxWords; w += 32) bits[w] = 0u;
      __syncwarp();
      for (int n = lane; n < cnt[0]; n += 32) {
        const int j = list[0][n];
        if (j >= 0 && j < s1) atomicOr(&bits[j >> 5], 1u << (j & 31));
      }
      __syncwarp();
      int uni = 0;  // entries of the second list not in the first
      for (int w = lane; w < kMaxWords; w += 32) uni += __popc(bits[w]);
      for (int n = lane; n < cnt[1]; n += 32) {
        const int j = list[1][n];
        if (j >= 0 && j < s1 && !((bits[j >> 5] >> (j & 31)) & 1u)) ++uni;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) uni += __shfl_xor_sync(0xffffffffu, uni, o);
      if (lane == 0) atomicAdd(&sc->total[c], (unsigned long long)uni);
      __syncwarp();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = 0;
    for (int c = 1; c < ncand; ++c)
      if (sc->total[c] < sc->total[best]) best = c;
    sc->chosen = sc->cand[best];
    const unsigned long long m = sc->total[best] / kSamples;
    sc->mean_union = m > 0 ? (int)m : 1;
  }
  __syncthreads();
  const int d = sc->chosen;
  if (mean_union) *mean_union = sc->mean_union;
  __syncthreads();  // the scratch is handed back to the pipeline after this
  return d;
}

// ---------------------------------------------------------------- host side
// [B, S, h, D] bf16 viewed as a 4-D tensor (D, h, S, B); box = 64 columns x `rows` tokens.
inline bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *ptr,
              const Shape &s, int rows) {
  cuuint64_t dims[4] = {(cuuint64_t)s.D, (cuuint64_t)s.h, (cuuint64_t)s.S, (cuuint64_t)s.B};
  cuuint64_t strides[3] = {(cuuint64_t)s.D * 2, (cuuint64_t)s.h * s.D * 2,
                           (cuuint64_t)s.S * s.h * s.D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tcattn
}  // namespace nabla
