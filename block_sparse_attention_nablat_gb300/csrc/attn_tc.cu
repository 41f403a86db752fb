// K3 -- bf16 block-sparse attention forward on the tcgen05 tensor cores.
//
// FastVideo API reference, page "nabla", NablaAttentionImpl.forward: softmax
// attention restricted to the kept 64x64 blocks of the NABLA block mask (full
// blocks, non-causal, default scale 1/sqrt(D)); gist.science NABLA summary,
// Methodology "Expansion".  The flex-attention kernel the page calls is prior
// art; this kernel is designed for sm_103a:
//
//  * Work unit = (batch, head, pair of adjacent query blocks): 128 query rows,
//    the M = 128 shape of a single-CTA tcgen05 MMA.  The unit walks the UNION
//    of the two blocks' kept-KV lists in ascending order; each entry carries
//    two membership bits, and rows of a block that did not keep an entry get
//    P = 0 for it (their softmax skips it).  Persistent CTAs (one per SM, the
//    kernel needs ~225 KB of shared memory and 384 TMEM columns) take units
//    round-robin in head-major order so concurrently running CTAs share one
//    head's K/V in L2.
//  * Warp roles: warp 0 builds the unit's entry bitmaps from kv_inds and issues
//    TMA loads (Q once per unit; K and V tiles of each kept block into a
//    6-deep ring); warp 1 (one thread) issues all MMAs; warps 4-7 (thread r =
//    TMEM lane r = query row r) run the online softmax and the epilogue.
//  * Per step (two KV entries): S = Q K^T as two 128x64 MMAs (K = D) into a
//    TMEM score buffer (two buffers, so QK of step s+1 overlaps the softmax of
//    step s); the softmax writes P back over the scores as packed bf16, and
//    PV accumulates O (128 x D fp32 in TMEM) with P taken straight from TMEM
//    as the A operand and V (MN-major) from shared memory.
//  * Online softmax in base 2 with the scale folded in; the running max is
//    only raised (and O, l rescaled) when it grows by more than 2^8, so the
//    O correction through TMEM is rare; the result is exact either way since
//    O and l always share the same reference max.
//  * Every mbarrier wait is bounded (1 s); on expiry the kernel records
//    NABLA_ERR_TIMEOUT, all roles stop, and TMEM is released.  Out-of-range or
//    unsorted kv_inds entries and out-of-range kv_nb are skipped and recorded
//    as NABLA_ERR_BAD_INDEX.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>

#include "internal.h"
#include "tc_ptx.cuh"

namespace nabla {
namespace {

using namespace tc;

constexpr int kMaxWords = 64;  // s1 <= 2048 blocks -> 64 bitmap words

struct UnitInfo {
  uint32_t a[kMaxWords];  // kept by the first query block of the pair
  uint32_t b[kMaxWords];  // kept by the second
  int n;                  // union size
  int pad;
};

template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;             // 64-column (128-byte) swizzle boxes
  static constexpr int kQBytes = 128 * D * 2;       // two query blocks
  static constexpr int kTileBytes = 64 * D * 2;     // one K or V block
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = D == 128 ? 6 : 12;
  static constexpr uint32_t kOCol = 0;              // O accumulator: TMEM columns [0, D)
  static constexpr uint32_t kSCol = 128;            // score buffers: [128, 256) and [256, 384)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescQK = idesc_bf16(128, 64, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, D, 0, 1);
  // shared-memory layout (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffStages = kQBytes;
  static constexpr int kOffInfo = kOffStages + kStages * kStageBytes;
  static constexpr int kOffBars = kOffInfo + 2 * (int)sizeof(UnitInfo);
  static constexpr int kNumBars = 2 * kStages + 14;
  static constexpr int kOffMisc = kOffBars + 8 * kNumBars;
  static constexpr int kSmemBytes = 1024 + kOffMisc + 16;
};

struct Bars {
  uint64_t *kv_full, *kv_empty, *q_full, *q_empty, *info_full, *info_empty, *s_full, *p_full,
      *pv_done, *o_free, *drain;
};

struct Cursor {
  int w;
  uint32_t m;
};

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

struct Params {
  __nv_bfloat16 *o;
  const int32_t *kv_nb, *kv_inds;
  int B, S, h;
  float scale_log2;
  int *status;
};

// On the abort path: wait (bounded, ignoring the abort flag) until the last
// copies this thread issued have landed, so none writes shared memory after exit.
template <int D>
__device__ void drain_copies(const Params &P, const Bars &bar, uint32_t ge, uint32_t kq,
                             bool q_loaded) {
  using C = Cfg<D>;
  const uint32_t first = ge > (uint32_t)C::kStages ? ge - C::kStages : 0u;
  for (uint32_t e = first; e < ge; ++e)
    mbar_wait(&bar.kv_full[e % C::kStages], (e / C::kStages) & 1u, nullptr, P.status,
              kDevTimeout);
  if (q_loaded && kq > 0) mbar_wait(bar.q_full, (kq - 1) & 1u, nullptr, P.status, kDevTimeout);
}

// Warp 0: entry bitmaps + TMA loads.
template <int D>
__device__ void producer(const Params &P, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                         const CUtensorMap *tmV, uint8_t *smem, UnitInfo *info, const Bars &bar,
                         volatile int *abort) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1, words = (s1 + 31) >> 5;
  const long units = (long)P.B * P.h * npairs;
  uint32_t ge = 0, kq = 0;
  int k = 0;
  for (long u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    __syncwarp();
    if (__shfl_sync(0xffffffffu, *abort, 0)) break;
    const int ub = k & 1;
    UnitInfo &inf = info[ub];
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&bar.info_empty[ub], ((k >> 1) & 1) ^ 1, abort, P.status, kDevTimeout);
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    const long bh = u / npairs;
    const int pr = (int)(u - bh * npairs);
    const int b = (int)(bh / P.h), hh = (int)(bh - (long)b * P.h);
    // ---- union of the two kept lists as bitmaps
    for (int w = lane; w < kMaxWords; w += 32) {
      inf.a[w] = 0u;
      inf.b[w] = 0u;
    }
    __syncwarp();
    bool bad = false;
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const int qb = 2 * pr + side;
      if (qb >= s1) break;
      const size_t row = (size_t)bh * s1 + qb;
      int cnt = P.kv_nb[row];
      if (cnt < 0 || cnt > s1) {
        bad = true;
        cnt = 0;
      }
      const int32_t *list = P.kv_inds + row * s1;
      uint32_t *bits = side ? inf.b : inf.a;
      for (int n = lane; n < cnt; n += 32) {
        const int j = list[n];
        const bool in_range = j >= 0 && j < s1;
        const bool sorted = n == 0 || list[n - 1] < j;
        if (in_range && sorted)
          atomicOr(&bits[j >> 5], 1u << (j & 31));
        else
          bad = true;
      }
    }
    if (bad) atomicCAS(P.status, kDevOk, kDevBadIndex);
    __syncwarp();
    int cnt = 0;
    for (int w = lane; w < words; w += 32) cnt += __popc(inf.a[w] | inf.b[w]);
#pragma unroll
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) inf.n = cnt;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.info_full[ub]);
    // ---- TMA loads (one thread)
    if (lane == 0 && cnt > 0) {
      bool go = mbar_wait(bar.q_empty, (kq & 1) ^ 1, abort, P.status, kDevTimeout);
      if (go) {
        mbar_expect_tx(bar.q_full, C::kQBytes);
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_4d(smem + C::kOffQ + c * 128 * 128, tmQ, bar.q_full, c * 64, hh, pr * 128, b);
      }
      ++kq;
      Cursor cur{0, inf.a[0] | inf.b[0]};
      for (int e = 0; go && e < cnt; ++e, ++ge) {
        if (*abort) {
          go = false;
          break;
        }
        uint32_t fl;
        const int j = next_entry(inf, cur, fl);
        const uint32_t st = ge % C::kStages, rnd = ge / C::kStages;
        if (!mbar_wait(&bar.kv_empty[st], (rnd & 1) ^ 1, abort, P.status, kDevTimeout)) {
          go = false;
          break;
        }
        uint8_t *kt = smem + C::kOffStages + st * C::kStageBytes;
        uint8_t *vt = kt + C::kTileBytes;
        mbar_expect_tx(&bar.kv_full[st], C::kStageBytes);
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c) {
          tma_load_4d(kt + c * 64 * 128, tmK, &bar.kv_full[st], c * 64, hh, j * 64, b);
          tma_load_4d(vt + c * 64 * 128, tmV, &bar.kv_full[st], c * 64, hh, j * 64, b);
        }
      }
    }
  }
  if (lane == 0 && *abort) drain_copies<D>(P, bar, ge, kq, true);
}

// Warp 1, lane 0: MMA issue.
template <int D>
__device__ void mma_issuer(const Params &P, uint8_t *smem, UnitInfo *info, const Bars &bar,
                           uint32_t tmem, volatile int *abort) {
  using C = Cfg<D>;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const uint32_t q_addr = smem_u32(smem + C::kOffQ);
  const uint32_t st_addr = smem_u32(smem + C::kOffStages);
  uint32_t ge = 0, gs = 0, kq = 0;
  int k = 0;
  for (long u = blockIdx.x; u < units && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&bar.info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) break;
    const int n = info[ub].n;
    const int steps = (n + 1) >> 1;
    if (steps > 0) {
      if (!mbar_wait(bar.q_full, kq & 1, abort, P.status, kDevTimeout)) break;
      tc_fence_after();
      bool ok = true;
      auto issue_qk = [&](int s) {
        const uint32_t g = gs + s, sb = g & 1u;
        ok = ok && mbar_wait(&bar.pv_done[sb], ((g >> 1) & 1u) ^ 1u, abort, P.status, kDevTimeout);
        for (int x = 0; x < 2 && ok; ++x) {
          const int e = 2 * s + x;
          if (e >= n) break;
          const uint32_t ee = ge + e, st = ee % C::kStages;
          ok = mbar_wait(&bar.kv_full[st], (ee / C::kStages) & 1u, abort, P.status, kDevTimeout);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + C::kSCol + sb * 128 + x * 64;
          const uint32_t kb = st_addr + st * C::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (uint32_t)(kk & 3) * 32u;  // 16-element step inside the 128-B atom
            const uint64_t a = smem_desc_sw128(q_addr + (kk >> 2) * 128 * 128 + koff, 16, 1024);
            const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * 64 * 128 + koff, 16, 1024);
            mma_ss(d, a, bd, C::kIdescQK, kk > 0 ? 1u : 0u);
          }
        }
        if (ok) mma_commit(&bar.s_full[sb]);
      };
      issue_qk(0);
      if (steps == 1 && ok) mma_commit(bar.q_empty);
      for (int s = 0; s < steps && ok; ++s) {
        if (s + 1 < steps) {
          issue_qk(s + 1);
          if (s + 2 == steps && ok) mma_commit(bar.q_empty);  // last QK of the unit issued
        }
        if (!ok) break;
        const uint32_t g = gs + s, sb = g & 1u;
        if (s == 0 && kq > 0) {
          ok = mbar_wait(bar.o_free, (kq - 1) & 1u, abort, P.status, kDevTimeout);
          if (!ok) break;
        }
        ok = mbar_wait(&bar.p_full[sb], (g >> 1) & 1u, abort, P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        for (int x = 0; x < 2; ++x) {
          const int e = 2 * s + x;
          if (e >= n) break;
          const uint32_t st = (ge + e) % C::kStages;
          const uint32_t vb = st_addr + st * C::kStageBytes + C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a = tmem + C::kSCol + sb * 128 + x * 32 + kk * 8;
            const uint64_t bd = smem_desc_sw128(vb + kk * 16 * 128, 64 * 128, 1024);
            mma_ts(tmem + C::kOCol, a, bd, C::kIdescPV, (s > 0 || x > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&bar.pv_done[sb]);
        for (int x = 0; x < 2; ++x) {
          const int e = 2 * s + x;
          if (e >= n) break;
          mma_commit(&bar.kv_empty[(ge + e) % C::kStages]);
        }
      }
      if (!ok) break;
      ++kq;
    }
    mbar_arrive(&bar.info_empty[ub]);
    ge += n;
    gs += steps;
  }
  // never release TMEM / exit with MMAs in flight (matters only on the abort path)
  mma_commit(bar.drain);
  mbar_wait(bar.drain, 0, nullptr, P.status, kDevTimeout);
}

// Warps 4-7: online softmax + epilogue.  Thread = TMEM lane = query row.
template <int D>
__device__ void softmax_epilogue(const Params &P, UnitInfo *info, const Bars &bar, uint32_t tmem,
                                 volatile int *abort) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = warp & 3;
  const int row = q4 * 32 + lane;
  const int half = row >> 6;
  const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const float sl2 = P.scale_log2;
  uint32_t gs = 0;
  int k = 0;
  for (long u = blockIdx.x; u < units && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&bar.info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) break;
    const UnitInfo &inf = info[ub];
    const int n = inf.n;
    const int steps = (n + 1) >> 1;
    const long bh = u / npairs;
    const int pr = (int)(u - bh * npairs);
    const int b = (int)(bh / P.h), hh = (int)(bh - (long)b * P.h);
    const int qb = 2 * pr + half;
    float m_run = -INFINITY, l_run = 0.f;
    Cursor cur{0, inf.a[0] | inf.b[0]};
    bool ok = true;
    for (int s = 0; s < steps; ++s) {
      const uint32_t g = gs + s, sb = g & 1u;
      uint32_t f0 = 0, f1 = 0;
      next_entry(inf, cur, f0);
      const bool has1 = 2 * s + 1 < n;
      if (has1) next_entry(inf, cur, f1);
      const bool act0 = (f0 >> half) & 1u;
      const bool act1 = has1 && ((f1 >> half) & 1u);
      ok = mbar_wait(&bar.s_full[sb], (g >> 1) & 1u, abort, P.status, kDevTimeout);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sbase = tmem + lane_base + C::kSCol + sb * 128;
      uint32_t r0[32], r1[32], r2[32], r3[32];
      if (act0) {
        tmem_ld32(sbase + 0, r0);
        tmem_ld32(sbase + 32, r1);
      }
      if (act1) {
        tmem_ld32(sbase + 64, r2);
        tmem_ld32(sbase + 96, r3);
      }
      tmem_wait_ld();
      if (act0) {
        reg_fence(r0);
        reg_fence(r1);
      }
      if (act1) {
        reg_fence(r2);
        reg_fence(r3);
      }
      // row max of the raw scores (the scale may be negative)
      float hi = -INFINITY, lo = INFINITY;
      if (act0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x0 = __uint_as_float(r0[i]), x1 = __uint_as_float(r1[i]);
          hi = fmaxf(hi, fmaxf(x0, x1));
          lo = fminf(lo, fminf(x0, x1));
        }
      }
      if (act1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x0 = __uint_as_float(r2[i]), x1 = __uint_as_float(r3[i]);
          hi = fmaxf(hi, fmaxf(x0, x1));
          lo = fminf(lo, fminf(x0, x1));
        }
      }
      const bool any = act0 || act1;
      if (any) {
        const float mx = sl2 >= 0.f ? hi * sl2 : lo * sl2;
        const float m_new = fmaxf(m_run, mx);
        const bool resc = m_run != -INFINITY && m_new > m_run + 8.0f;
        if (__any_sync(0xffffffffu, resc)) {
          // O must hold every PV up to the previous step before it is rescaled
          const uint32_t gp = g - 1;
          ok = mbar_wait(&bar.pv_done[gp & 1u], (gp >> 1) & 1u, abort, P.status, kDevTimeout);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = resc ? ex2(m_run - m_new) : 1.0f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t t[32];
            tmem_ld32(tmem + lane_base + C::kOCol + c * 32, t);
            tmem_wait_ld();
            reg_fence(t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st32(tmem + lane_base + C::kOCol + c * 32, t);
          }
          tmem_wait_st();
          if (resc) {
            l_run *= alpha;
            m_run = m_new;
          }
        }
        if (m_run == -INFINITY) m_run = m_new;
      }
      // P = 2^(s * scale * log2 e - m), packed bf16 pairs, over the score columns
      float lsum = 0.f;
      uint32_t pk[32];
      if (act0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = ex2(fmaf(__uint_as_float(r0[2 * i]), sl2, -m_run));
          const float a1 = ex2(fmaf(__uint_as_float(r0[2 * i + 1]), sl2, -m_run));
          const float b0 = ex2(fmaf(__uint_as_float(r1[2 * i]), sl2, -m_run));
          const float b1 = ex2(fmaf(__uint_as_float(r1[2 * i + 1]), sl2, -m_run));
          lsum += (a0 + a1) + (b0 + b1);
          pk[i] = pack_bf16x2(a0, a1);
          pk[16 + i] = pack_bf16x2(b0, b1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = 0u;
      }
      tmem_st32(sbase + 0, pk);
      if (has1) {
        if (act1) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = ex2(fmaf(__uint_as_float(r2[2 * i]), sl2, -m_run));
            const float a1 = ex2(fmaf(__uint_as_float(r2[2 * i + 1]), sl2, -m_run));
            const float b0 = ex2(fmaf(__uint_as_float(r3[2 * i]), sl2, -m_run));
            const float b1 = ex2(fmaf(__uint_as_float(r3[2 * i + 1]), sl2, -m_run));
            lsum += (a0 + a1) + (b0 + b1);
            pk[i] = pack_bf16x2(a0, a1);
            pk[16 + i] = pack_bf16x2(b0, b1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = 0u;
        }
        tmem_st32(sbase + 32, pk);
      }
      l_run += lsum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar.p_full[sb]);
    }
    if (!ok) break;
    // ---- epilogue: O / l -> bf16 -> o[b, qb*64 + r, hh, :]
    if (steps > 0) {
      const uint32_t gl = gs + steps - 1;
      ok = mbar_wait(&bar.pv_done[gl & 1u], (gl >> 1) & 1u, abort, P.status, kDevTimeout);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
    }
    const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
    const bool row_valid = qb < s1;
    __nv_bfloat16 *orow =
        P.o + (((size_t)b * P.S + (size_t)qb * 64 + (row & 63)) * P.h + hh) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t t[32];
      if (steps > 0) {
        tmem_ld32(tmem + lane_base + C::kOCol + c * 32, t);
        tmem_wait_ld();
        reg_fence(t);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) t[i] = 0u;
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(t[2 * i]) * inv, __uint_as_float(t[2 * i + 1]) * inv);
      if (row_valid) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
      }
    }
    tc_fence_before();
    if (steps > 0) mbar_arrive(bar.o_free);
    mbar_arrive(&bar.info_empty[ub]);
    gs += steps;
  }
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, Params P) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  UnitInfo *info = reinterpret_cast<UnitInfo *>(smem + C::kOffInfo);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
  Bars bar;
  bar.kv_full = bars;
  bar.kv_empty = bars + C::kStages;
  bar.q_full = bars + 2 * C::kStages;
  bar.q_empty = bar.q_full + 1;
  bar.info_full = bar.q_full + 2;
  bar.info_empty = bar.q_full + 4;
  bar.s_full = bar.q_full + 6;
  bar.p_full = bar.q_full + 8;
  bar.pv_done = bar.q_full + 10;
  bar.o_free = bar.q_full + 12;
  bar.drain = bar.q_full + 13;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bar.kv_full[i], 1);
      mbar_init(&bar.kv_empty[i], 1);
    }
    mbar_init(bar.q_full, 1);
    mbar_init(bar.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.info_full[i], 1);
      mbar_init(&bar.info_empty[i], 128 + 1);
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.p_full[i], 128);
      mbar_init(&bar.pv_done[i], 1);
    }
    mbar_init(bar.o_free, 128);
    mbar_init(bar.drain, 1);
    *abort = 0;
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    producer<D>(P, &tmQ, &tmK, &tmV, smem, info, bar, abort);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D>(P, smem, info, bar, tmem, abort);
    __syncwarp();
  } else if (warp >= 4) {
    softmax_epilogue<D>(P, info, bar, tmem, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode(cudaError_t *err) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    *err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                            cudaEnableDefault, &q);
    if (*err != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
      if (*err == cudaSuccess) *err = cudaErrorNotSupported;
      return nullptr;
    }
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *err = cudaSuccess;
  return fn;
}

// [B, S, h, D] bf16 viewed as a 4-D tensor (D, h, S, B); box = 64 columns x `rows` tokens.
bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *ptr,
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

template <int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, const Shape &s,
                     const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                     int *status, cudaStream_t st) {
  using C = Cfg<D>;
  cudaError_t err;
  auto enc = get_encode(&err);
  if (!enc) return err;
  CUtensorMap mq, mk, mv;
  if (!make_map(enc, &mq, q, s, 128) || !make_map(enc, &mk, k, s, 64) ||
      !make_map(enc, &mv, v, s, 64))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  auto kern = attn_tc_kernel<D>;
  if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  C::kSmemBytes)) != cudaSuccess)
    return err;
  const long units = (long)s.B * s.h * ((s.s1 + 1) / 2);
  const int grid = (int)(units < sms ? units : sms);
  Params p{static_cast<__nv_bfloat16 *>(o), kv_nb, kv_inds, s.B, s.S, s.h,
           scale * 1.4426950408889634f, status};
  kern<<<grid, 256, C::kSmemBytes, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const void *q, const void *k, const void *v, const Shape &s,
                           const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                           int *status, cudaStream_t st) {
  if (s.D == 64) return launch_d<64>(q, k, v, s, kv_nb, kv_inds, scale, o, status, st);
  return launch_d<128>(q, k, v, s, kv_nb, kv_inds, scale, o, status, st);
}

}  // namespace nabla
