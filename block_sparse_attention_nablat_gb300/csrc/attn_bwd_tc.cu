// K7t -- bf16 block-sparse attention backward on the tcgen05 tensor cores.
//
// gist.science NABLA summary, "Dual-Phase Acceleration" and Experimental
// Results (training with the block mask); FastVideo API reference, page
// "nabla", NablaAttentionImpl.forward is the function differentiated.  With
// z = scale q k^T over a row's kept tokens, P = softmax(z) = 2^(z log2(e) -
// lse2), delta_s = dout_s . o_s and dz = P (dout v^T - delta):
//   dV = P^T dout,  dK = scale dz^T q,  dQ = scale dz k.
//
// One kernel template, two modes over the same step:
//  * kDQ = false (dK, dV): unit = (batch, head, pair of KEY blocks at the
//    in-kernel stride); its entries are the query blocks that kept either key
//    block (the transposed lists), ascending.  The pair's K and V rows are the
//    A operands, loaded once per unit; each step loads the entry's q and dout
//    tiles and its 64 lse2 / delta values.
//  * kDQ = true (dQ): unit = (batch, head, pair of QUERY blocks); entries =
//    the key blocks either block kept.  A operands = the pair's q and dout
//    rows; each step loads the entry's k and v tiles; lse2 / delta are per row.
// A step (64 entry rows) issues two SS MMAs, X = A1 T1^T and Y = A2 T2^T
// (M = 128, N = 64), into one of two TMEM buffers.  Warps 4-11 (thread = TMEM
// lane = row of the unit pair; warps 4-7 take entry columns 0-31, warps 8-11
// columns 32-63) load their X and Y columns and form
//   dK/dV: P^T = 2^(X sl2 - lse2[col]),  dz^T = P^T (Y - delta[col]);
//   dQ:    P   = 2^(X sl2 - lse2[row]),  dz   = P   (Y - delta[row]);
// with P = 0 in the rows whose block did not keep the entry (the producer warp
// lists each entry's membership bits once per unit, so the softmax threads
// read one byte per entry instead of scanning the bitmaps).  P and dz are
// stored as bf16 and TS MMAs accumulate
//   dK/dV: dV += P^T dout, dK += dz^T q;   dQ: dQ += dz k.
// One thread (warp 1) issues the SS MMAs and another (warp 2) the TS MMAs, so
// a wait in one stream never holds back the other; with two X / Y buffers,
// SS(g+1) depends on step g-1 only, so the tensor pipe works on TS(g-1) and
// SS(g+1) while the softmax of step g runs.  TMEM (512
// columns):
//   dK/dV: dK [0, D), dV [D, 2D), buffer b at 2D + 128 b (X in its first 64
//          columns, Y in the next 64).  P and dz are written in place over the
//          columns each group has read (group g: P at X + 32 g, dz at Y + 32 g,
//          16 columns each), and SS(g+2) waits until TS(g) has read them;
//   dQ:    dQ [0, D), buffer b at D + 128 b, dz buffer b at D + 256 + 64 b; the
//          softmax releases X / Y as soon as it has loaded them, and writes dz
//          once TS(g-2) has read the dz buffer.
// Every mbarrier wait is bounded
// (1 s); on expiry the kernel records NABLA_ERR_TIMEOUT, the roles stop,
// in-flight copies and MMAs are drained and TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "tc_ptx.cuh"

namespace nabla {
namespace {

using namespace tc;
using namespace tcattn;

template <int D, bool kDQ>
struct BCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kPairBytes = 128 * D * 2;  // A operand: 128 rows
  static constexpr int kTileBytes = 64 * D * 2;   // one 64-row tile
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;  // T1, T2, lse2 / delta (dK/dV)
  static constexpr int kOffA1 = 0;
  static constexpr int kOffA2 = kPairBytes;
  static constexpr int kOffStage = 2 * kPairBytes;
  static constexpr int kOffInfo = kOffStage + kStages * kStageBytes;
  static constexpr int kOffFlags = kOffInfo + 2 * (int)sizeof(UnitInfo);  // [2][kMaxEntries]
  static constexpr int kOffBars = kOffFlags + 2 * kMaxEntries;
  static constexpr uint32_t kAcc1 = 0, kAcc0 = D;
  static constexpr uint32_t kXY = kDQ ? D : 2 * D;  // X / Y buffer b at kXY + 128 b
  static constexpr uint32_t kPD = D + 256;          // dQ: dz buffer b at kPD + 64 b
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdSS = idesc_bf16(128, 64, 0, 0);
  static constexpr uint32_t kIdTS = idesc_bf16(128, D, 0, 1);
  static constexpr int kThreads = 384;
  static constexpr int kSoftmax = 256;  // threads of warps 4-11
  static_assert(kXY + 256 <= kTmemCols && (!kDQ || kPD + 128 <= kTmemCols), "TMEM budget");
};

struct BSync {
  uint64_t st_full[4], st_empty[4], x_free[4];  // x_free: dK/dV, the TS MMAs that read P are done
  uint64_t a_full, a_empty, info_full[2], info_empty[2];
  uint64_t s_full[2], x_read[2], p_full[2];
  uint64_t acc_full, acc_free, drain;
  uint32_t tmem_slot;
  int abort;
};

template <int D>
constexpr int bwd_smem_bytes() {
  return 1024 + BCfg<D, false>::kOffBars + (int)sizeof(BSync);
}
static_assert(bwd_smem_bytes<128>() <= 232448, "shared memory budget (D=128)");
static_assert(BCfg<128, false>::kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
static_assert(BCfg<64, false>::kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");

struct TcParams {
  __nv_bfloat16 *out1, *out0;      // dK/dV mode: dK, dV; dQ mode: dQ, null
  const int32_t *kv_nb, *kv_inds;  // the units' lists (transposed for dK/dV)
  const float *lse2, *delta;       // [B, h, S]
  int B, S, h;
  float scale_log2, scale;
  int *status;
  int pstride;
};

// Warp 0: entry bitmaps of every unit, TMA loads of the unit's A rows and of
// every entry's tiles (+ the entry's lse2 / delta in dK/dV mode).
template <int D, bool kDQ>
__device__ void b_producer(const TcParams &P, const CUtensorMap *mA1, const CUtensorMap *mA2,
                           const CUtensorMap *mT1, const CUtensorMap *mT2, uint8_t *smem,
                           UnitInfo *info, BSync *sy, volatile int *abort) {
  using C = BCfg<D, kDQ>;
  const int lane = threadIdx.x & 31;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  uint32_t ge = 0, ka = 0;
  bool go = true;
  int k = 0;
  for (long u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    __syncwarp();
    if (__shfl_sync(0xffffffffu, (!go || *abort) ? 1 : 0, 0)) break;
    const int ub = k & 1;
    UnitInfo &inf = info[ub];
    bool ok = true;
    if (lane == 0)
      ok = mbar_wait(&sy->info_empty[ub], ((k >> 1) & 1) ^ 1, abort, P.status, kDevTimeout);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    const Unit un = decode(u, npairs, P.h);
    const long bh = (long)un.b * P.h + un.hh;
    for (int w = lane; w < kMaxWords; w += 32) {
      inf.a[w] = 0u;
      inf.b[w] = 0u;
    }
    __syncwarp();
    bool bad = false;
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const int blk = pair_block(un.pr, side, P.pstride);
      if (blk >= s1) break;
      const size_t row = (size_t)bh * s1 + blk;
      int cnt = P.kv_nb[row];
      if (cnt < 0 || cnt > s1) {
        bad = true;
        cnt = 0;
      }
      const int32_t *list = P.kv_inds + row * s1;
      uint32_t *bits = side ? inf.b : inf.a;
      for (int n = lane; n < cnt; n += 32) {
        const int j = list[n];
        if (j >= 0 && j < s1 && (n == 0 || list[n - 1] < j))
          atomicOr(&bits[j >> 5], 1u << (j & 31));
        else
          bad = true;
      }
    }
    if (bad) atomicCAS(P.status, kDevOk, kDevBadIndex);
    __syncwarp();
    // entry count, and the entries' membership bits for the softmax warps
    const int cnt = list_entries(inf, smem + C::kOffFlags + ub * kMaxEntries, lane);
    if (lane == 0) inf.n = cnt;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sy->info_full[ub]);
    if (cnt == 0) continue;
    // ---- the unit's A rows (a block past s1 is zero-filled)
    if (lane == 0) {
      go = mbar_wait(&sy->a_empty, (ka & 1) ^ 1, abort, P.status, kDevTimeout);
      if (go) {
        mbar_expect_tx(&sy->a_full, 2 * C::kPairBytes);
#pragma unroll
        for (int side = 0; side < 2; ++side)
#pragma unroll
          for (int c = 0; c < C::kBoxes; ++c) {
            const int blk = pair_block(un.pr, side, P.pstride) * 64;
            tma_load_4d(smem + C::kOffA1 + c * 128 * 128 + side * 64 * 128, mA1, &sy->a_full,
                        c * 64, un.hh, blk, un.b);
            tma_load_4d(smem + C::kOffA2 + c * 128 * 128 + side * 64 * 128, mA2, &sy->a_full,
                        c * 64, un.hh, blk, un.b);
          }
        ++ka;
      }
    }
    go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
    if (!go) break;
    // ---- the entries' tiles, in entry order
    Cursor cur{0, inf.a[0] | inf.b[0]};
    for (int e = 0; e < cnt && go; ++e, ++ge) {
      const uint32_t st = ge % C::kStages;
      if (lane == 0)
        go = mbar_wait(&sy->st_empty[st], ((ge / C::kStages) & 1) ^ 1, abort, P.status,
                       kDevTimeout);
      go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
      if (!go) break;
      uint32_t fl;
      const int j = next_entry(inf, cur, fl);
      uint8_t *stage = smem + C::kOffStage + st * C::kStageBytes;
      if (lane == 0) {
        mbar_expect_tx(&sy->st_full[st], 2 * C::kTileBytes + (kDQ ? 0 : 512));
        if (!kDQ) {  // the entry's 64 lse2 and 64 delta values (16-byte aligned rows)
          const size_t at = (size_t)bh * P.S + (size_t)j * 64;
          bulk_load(stage + 2 * C::kTileBytes, P.lse2 + at, 256, &sy->st_full[st]);
          bulk_load(stage + 2 * C::kTileBytes + 256, P.delta + at, 256, &sy->st_full[st]);
        }
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c) {
          tma_load_4d(stage + c * 64 * 128, mT1, &sy->st_full[st], c * 64, un.hh, j * 64, un.b);
          tma_load_4d(stage + C::kTileBytes + c * 64 * 128, mT2, &sy->st_full[st], c * 64,
                      un.hh, j * 64, un.b);
        }
      }
    }
  }
  if (lane == 0 && (!go || *abort)) {  // let in-flight copies land before the CTA exits
    for (uint32_t e = ge > (uint32_t)C::kStages ? ge - C::kStages : 0u; e < ge; ++e)
      mbar_wait(&sy->st_full[e % C::kStages], (e / C::kStages) & 1u, nullptr, P.status,
                kDevTimeout);
    if (ka > 0) mbar_wait(&sy->a_full, (ka - 1) & 1u, nullptr, P.status, kDevTimeout);
  }
}

// Warp 1, lane 0: the SS MMAs.  SS(g) once its stage has landed and buffer
// g & 1 is free again (dQ: the softmax of step g-2 has read X / Y; dK/dV: the
// TS MMAs of step g-2 have read the P / dz written over them).
template <int D, bool kDQ>
__device__ void b_ss(const TcParams &P, uint8_t *smem, UnitInfo *info, BSync *sy, uint32_t tmem,
                     volatile int *abort) {
  using C = BCfg<D, kDQ>;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const uint64_t a1_desc = smem_desc_sw128(smem_u32(smem + C::kOffA1), 16, 1024);
  const uint64_t a2_desc = smem_desc_sw128(smem_u32(smem + C::kOffA2), 16, 1024);
  const uint64_t tk_desc = smem_desc_sw128(smem_u32(smem + C::kOffStage), 16, 1024);
  uint32_t g = 0, ge = 0, ka = 0;
  bool ok = true;
  int k = 0;
  for (long u = blockIdx.x; u < units && ok && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&sy->info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) break;
    const int n = info[ub].n;
    if (n > 0) {
      if (!mbar_wait(&sy->a_full, ka & 1u, abort, P.status, kDevTimeout)) break;
      for (int e = 0; e < n; ++e, ++g, ++ge) {
        const uint32_t st = ge % C::kStages;
        const uint32_t b = g & 1u;
        ok = mbar_wait(&sy->st_full[st], (ge / C::kStages) & 1u, abort, P.status, kDevTimeout);
        const uint32_t g2 = g - 2;
        // dQ: the softmax of step g-2 has read X / Y.  dK/dV: P and dz of step g-2 sit
        // over X and Y; X may be rewritten once the TS MMAs that read P (dV) are done
        // (x_free), Y once those that read dz (dK) are done too (st_empty)
        if (ok && g >= 2)
          ok = kDQ ? mbar_wait(&sy->x_read[b], ((g >> 1) - 1) & 1u, abort, P.status, kDevTimeout)
                   : mbar_wait(&sy->x_free[g2 % C::kStages], (g2 / C::kStages) & 1u, abort,
                               P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        const uint64_t t1 = tk_desc + (uint64_t)((st * C::kStageBytes) >> 4);
        const uint64_t t2 = tk_desc + (uint64_t)((st * C::kStageBytes + C::kTileBytes) >> 4);
        const uint32_t xb = tmem + C::kXY + b * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t da = (uint64_t)((((kk >> 2) * 128 * 128) + (kk & 3) * 32) >> 4);
          const uint64_t dt = (uint64_t)((((kk >> 2) * 64 * 128) + (kk & 3) * 32) >> 4);
          mma_ss(xb, a1_desc + da, t1 + dt, C::kIdSS, kk > 0 ? 1u : 0u);  // X = A1 T1^T
        }
        if (!kDQ && g >= 2) {
          ok = mbar_wait(&sy->st_empty[g2 % C::kStages], (g2 / C::kStages) & 1u, abort, P.status,
                         kDevTimeout);
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t da = (uint64_t)((((kk >> 2) * 128 * 128) + (kk & 3) * 32) >> 4);
          const uint64_t dt = (uint64_t)((((kk >> 2) * 64 * 128) + (kk & 3) * 32) >> 4);
          mma_ss(xb + 64, a2_desc + da, t2 + dt, C::kIdSS, kk > 0 ? 1u : 0u);  // Y = A2 T2^T
        }
        mma_commit(&sy->s_full[b]);
      }
      if (!ok) break;
      mma_commit(&sy->a_empty);  // the unit's A rows are no longer read
      ++ka;
    }
    mbar_arrive(&sy->info_empty[ub]);
  }
  mma_commit(&sy->drain);  // never exit with MMAs in flight
  mbar_wait(&sy->drain, 0, nullptr, P.status, kDevTimeout);
}

// Warp 2, lane 0: the TS MMAs.  TS(g) once the softmax of step g has written
// its P / dz (and, for a unit's first step, once the epilogue has read the
// previous unit's accumulators).  Its own issue stream, so a wait here never
// holds back the next SS MMAs.
template <int D, bool kDQ>
__device__ void b_ts(const TcParams &P, uint8_t *smem, UnitInfo *info, BSync *sy, uint32_t tmem,
                     volatile int *abort) {
  using C = BCfg<D, kDQ>;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const uint64_t tm_desc = smem_desc_sw128(smem_u32(smem + C::kOffStage), 64 * 128, 1024);
  uint32_t g = 0, ge = 0, ku = 0;
  bool ok = true;
  int k = 0;
  for (long u = blockIdx.x; u < units && ok && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&sy->info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) break;
    const int n = info[ub].n;
    if (n > 0) {
      for (int e = 0; e < n; ++e, ++g, ++ge) {
        const uint32_t st = ge % C::kStages;
        const uint32_t b = g & 1u;
        ok = mbar_wait(&sy->p_full[b], (g >> 1) & 1u, abort, P.status, kDevTimeout);
        if (ok && e == 0 && ku > 0)
          ok = mbar_wait(&sy->acc_free, (ku - 1) & 1u, abort, P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        const uint64_t t1 = tm_desc + (uint64_t)((st * C::kStageBytes) >> 4);
        const uint64_t t2 = tm_desc + (uint64_t)((st * C::kStageBytes + C::kTileBytes) >> 4);
        if (kDQ) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 16 entry rows per MMA
            const uint64_t dk = (uint64_t)((kk * 16 * 128) >> 4);
            const uint32_t acc = (e > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + C::kAcc1, tmem + C::kPD + b * 64 + kk * 8, t1 + dk, C::kIdTS, acc);
          }
        } else {
          // entries 32 g .. 32 g + 31 sit at columns 32 g .. 32 g + 15 of X and Y; the
          // MMAs that read P (in X) go first, so that X is free again sooner
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t xb = tmem + C::kXY + b * 128 + (kk >> 1) * 32 + (kk & 1) * 8;
            mma_ts(tmem + C::kAcc0, xb, t2 + (uint64_t)((kk * 16 * 128) >> 4), C::kIdTS,
                   (e > 0 || kk > 0) ? 1u : 0u);  // dV += P^T dout
          }
          mma_commit(&sy->x_free[st]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t xb = tmem + C::kXY + b * 128 + (kk >> 1) * 32 + (kk & 1) * 8;
            mma_ts(tmem + C::kAcc1, xb + 64, t1 + (uint64_t)((kk * 16 * 128) >> 4), C::kIdTS,
                   (e > 0 || kk > 0) ? 1u : 0u);  // dK += dz^T q
          }
        }
        // the stage (read by both streams; SS(g) finished before the softmax of
        // step g began) and the P / dz of buffer b are free once these are done:
        // one commit signals both (the stage ring and the steps count alike)
        mma_commit(&sy->st_empty[st]);
      }
      if (!ok) break;
      mma_commit(&sy->acc_full);
      ++ku;
    }
    mbar_arrive(&sy->info_empty[ub]);
  }
  mma_commit(&sy->drain);
  mbar_wait(&sy->drain, 0, nullptr, P.status, kDevTimeout);
}

// 32 columns of P and dz from X and Y (fp32 in registers), stored as bf16 over
// 16 TMEM columns each (P at paddr, dz at daddr).  lse / dl: per column (dK/dV)
// or the row's (dQ).
template <bool kDQ>
__device__ __forceinline__ void form_pd(const uint32_t (&x)[32], const uint32_t (&y)[32],
                                        const float *lse_c, const float *dl_c, float lse_r,
                                        float dl_r, float sl2, bool act, uint32_t paddr,
                                        uint32_t daddr) {
  uint32_t pk[16], dk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float p0 = 0.f, p1 = 0.f, d0 = 0.f, d1 = 0.f;
    if (act) {
      const float l0 = kDQ ? lse_r : lse_c[2 * i], l1 = kDQ ? lse_r : lse_c[2 * i + 1];
      const float e0 = kDQ ? dl_r : dl_c[2 * i], e1 = kDQ ? dl_r : dl_c[2 * i + 1];
      p0 = ex2(fmaf(__uint_as_float(x[2 * i]), sl2, -l0));
      p1 = ex2(fmaf(__uint_as_float(x[2 * i + 1]), sl2, -l1));
      d0 = p0 * (__uint_as_float(y[2 * i]) - e0);
      d1 = p1 * (__uint_as_float(y[2 * i + 1]) - e1);
    }
    pk[i] = pack_bf16x2(p0, p1);
    dk[i] = pack_bf16x2(d0, d1);
  }
  if (!kDQ) tmem_st16(paddr, pk);
  tmem_st16(daddr, dk);
}

// Warps 4-11: P and dz of every step (group grp = entry columns 32 grp ..
// 32 grp + 31), then the unit's gradient rows (group grp writes half of the D
// columns).
template <int D, bool kDQ>
__device__ void b_softmax(const TcParams &P, uint8_t *smem, UnitInfo *info, BSync *sy,
                          uint32_t tmem, volatile int *abort) {
  using C = BCfg<D, kDQ>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = (warp - 4) >> 2;
  const int q4 = warp & 3;
  const int row = q4 * 32 + lane;
  const int side = row >> 6;
  const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const float sl2 = P.scale_log2;
  uint32_t g = 0, ge = 0, ku = 0;
  bool live = true;
  int k = 0;
  for (long u = blockIdx.x; u < units && live; u += gridDim.x, ++k) {
    const int ub = k & 1;
    live = mbar_wait(&sy->info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout);
    if (!live) break;
    const int n = info[ub].n;
    const Unit un = decode(u, npairs, P.h);
    const long bh = (long)un.b * P.h + un.hh;
    const int blk = pair_block(un.pr, side, P.pstride);  // this thread's row block
    float lse_r = 0.f, dl_r = 0.f;
    if (kDQ && blk < s1 && n > 0) {
      lse_r = P.lse2[(size_t)bh * P.S + (size_t)blk * 64 + (row & 63)];
      dl_r = P.delta[(size_t)bh * P.S + (size_t)blk * 64 + (row & 63)];
    }
    // each entry's membership bits, listed by the producer
    const uint8_t *elist = smem + C::kOffFlags + ub * kMaxEntries;
    for (int e = 0; e < n && live; ++e, ++g, ++ge) {
      const uint32_t b = g & 1u, st = ge % C::kStages;
      const uint32_t fl = elist[e];
      const bool act = ((fl >> side) & 1u) != 0u;
      live = __all_sync(0xffffffffu,
                        mbar_wait(&sy->s_full[b], (g >> 1) & 1u, abort, P.status, kDevTimeout));
      if (!kDQ && live)  // the stage's lse2 / delta (bulk copies on st_full)
        live = __all_sync(0xffffffffu, mbar_wait(&sy->st_full[st], (ge / C::kStages) & 1u,
                                                 abort, P.status, kDevTimeout));
      if (!live) break;
      tc_fence_after();
      uint32_t x[32], y[32];
      const uint32_t xb = tmem + lane_base + C::kXY + b * 128;
      tmem_ld32(xb + grp * 32, x);
      tmem_ld32(xb + 64 + grp * 32, y);
      tmem_wait_ld();
      reg_fence(x);
      reg_fence(y);
      const float *ld = reinterpret_cast<const float *>(smem + C::kOffStage + st * C::kStageBytes +
                                                        2 * C::kTileBytes);
      if (kDQ) {
        tc_fence_before();
        mbar_arrive(&sy->x_read[b]);  // buffer b may take the products of step g + 2
        // the dz buffer of step g was last read by the TS MMAs of step g - 2, whose
        // completion st_empty[(g - 2) % 4] signals
        if (g >= 2) {
          const uint32_t g2 = g - 2;
          live = __all_sync(0xffffffffu, mbar_wait(&sy->st_empty[g2 % C::kStages],
                                                   (g2 / C::kStages) & 1u, abort, P.status,
                                                   kDevTimeout));
        }
        if (!live) break;
        tc_fence_after();
        const uint32_t pd = tmem + lane_base + C::kPD + b * 64;
        form_pd<kDQ>(x, y, ld, ld + 64, lse_r, dl_r, sl2, act, pd + grp * 16, pd + grp * 16);
      } else {  // in place over the 32 columns of X and Y this thread has just read
        form_pd<kDQ>(x, y, ld + grp * 32, ld + 64 + grp * 32, lse_r, dl_r, sl2, act,
                     xb + grp * 32, xb + 64 + grp * 32);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sy->p_full[b]);
    }
    if (!live) break;
    // ---- the unit's gradient rows: dK (scaled) and dV, or dQ (scaled); zero rows
    // for a unit with no entry
    if (n > 0) {
      live = __all_sync(0xffffffffu,
                        mbar_wait(&sy->acc_full, ku & 1u, abort, P.status, kDevTimeout));
      if (!live) break;
      tc_fence_after();
    }
    const bool row_ok = blk < s1;
    const size_t orow = (((size_t)un.b * P.S + (size_t)blk * 64 + (row & 63)) * P.h + un.hh) * D;
#pragma unroll 1
    for (int which = 0; which < (kDQ ? 1 : 2); ++which) {
      __nv_bfloat16 *dst = which ? P.out0 : P.out1;
      const float mul = which ? 1.0f : P.scale;
      const uint32_t col = which ? C::kAcc0 : C::kAcc1;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        const int c = grp * (D / 32) + cc;  // this group's 16-column pieces
        uint32_t t[16];
        if (n > 0) {
          tmem_ld16(tmem + lane_base + col + c * 16, t);
          tmem_wait_ld();
          reg_fence16(t);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] = 0u;
        }
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = pack_bf16x2(__uint_as_float(t[2 * i]) * mul, __uint_as_float(t[2 * i + 1]) * mul);
        if (row_ok) {
          uint4 *o = reinterpret_cast<uint4 *>(dst + orow + c * 16);
          o[0] = make_uint4(w[0], w[1], w[2], w[3]);
          o[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    if (n > 0) {
      tc_fence_before();
      mbar_arrive(&sy->acc_free);
      ++ku;
    }
    mbar_arrive(&sy->info_empty[ub]);  // done with this unit's bitmaps
  }
}

template <int D, bool kDQ>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap mA1,
                       const __grid_constant__ CUtensorMap mA2,
                       const __grid_constant__ CUtensorMap mT1,
                       const __grid_constant__ CUtensorMap mT2, TcParams P) {
  using C = BCfg<D, kDQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  UnitInfo *info = reinterpret_cast<UnitInfo *>(smem + C::kOffInfo);
  BSync *sy = reinterpret_cast<BSync *>(smem + C::kOffBars);
  volatile int *abort = &sy->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&sy->st_full[i], 1);
      mbar_init(&sy->st_empty[i], 1);
      mbar_init(&sy->x_free[i], 1);
    }
    mbar_init(&sy->a_full, 1);
    mbar_init(&sy->a_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sy->info_full[i], 1);
      mbar_init(&sy->info_empty[i], C::kSoftmax + 2);  // softmax threads + both MMA issuers
      mbar_init(&sy->p_full[i], C::kSoftmax);
      mbar_init(&sy->s_full[i], 1);
      mbar_init(&sy->x_read[i], C::kSoftmax);
    }
    mbar_init(&sy->acc_full, 1);
    mbar_init(&sy->acc_free, C::kSoftmax);
    mbar_init(&sy->drain, 2);  // one commit per MMA-issuing thread
    sy->abort = 0;
    tma_prefetch_desc(&mA1);
    tma_prefetch_desc(&mA2);
    tma_prefetch_desc(&mT1);
    tma_prefetch_desc(&mT2);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sy->tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sy->tmem_slot;
  pdl_wait();  // lists, lse2 / delta and the inputs are written
  static_assert(sizeof(StrideScratch) <= (size_t)C::kOffInfo - C::kOffStage, "scratch fits");
  TcParams Pp = P;
  Pp.pstride = choose_pair_stride(P, reinterpret_cast<StrideScratch *>(smem + C::kOffStage));

  if (warp == 0) {
    b_producer<D, kDQ>(Pp, &mA1, &mA2, &mT1, &mT2, smem, info, sy, abort);
  } else if (warp == 1) {
    if (lane == 0) b_ss<D, kDQ>(Pp, smem, info, sy, tmem, abort);
    __syncwarp();
  } else if (warp == 2) {
    if (lane == 0) b_ts<D, kDQ>(Pp, smem, info, sy, tmem, abort);
    __syncwarp();
  } else if (warp >= 4) {
    b_softmax<D, kDQ>(Pp, smem, info, sy, tmem, abort);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool kDQ>
cudaError_t launch_mode(const void *a1, const void *a2, const void *t1, const void *t2,
                        const Shape &s, TcParams p, cudaStream_t st) {
  using C = BCfg<D, kDQ>;
  cudaError_t err;
  auto enc = tensor_map_encoder(&err);
  if (!enc) return err;
  CUtensorMap m1, m2, m3, m4;
  if (!make_map(enc, &m1, a1, s, 64) || !make_map(enc, &m2, a2, s, 64) ||
      !make_map(enc, &m3, t1, s, 64) || !make_map(enc, &m4, t2, s, 64))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  auto kern = attn_bwd_tc_kernel<D, kDQ>;
  if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  bwd_smem_bytes<D>())) != cudaSuccess)
    return err;
  const long units = (long)s.B * s.h * ((s.s1 + 1) / 2);
  const int grid = (int)(units < sms ? units : sms);
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), bwd_smem_bytes<D>(), st, m1, m2, m3, m4,
                    p);
}

template <int D>
cudaError_t launch_both(const void *q, const void *k, const void *v, const void *dout,
                        const Shape &s, const int32_t *kv_nb, const int32_t *kv_inds,
                        const int32_t *qt_nb, const int32_t *qt_inds, const float *lse2,
                        const float *delta, float scale, void *dq, void *dk, void *dv,
                        int *status, cudaStream_t st) {
  const float sl2 = scale * 1.4426950408889634f;
  TcParams pkv{static_cast<__nv_bfloat16 *>(dk), static_cast<__nv_bfloat16 *>(dv), qt_nb, qt_inds,
               lse2, delta, s.B, s.S, s.h, sl2, scale, status, 1};
  cudaError_t e = launch_mode<D, false>(k, v, q, dout, s, pkv, st);
  if (e != cudaSuccess) return e;
  TcParams pq{static_cast<__nv_bfloat16 *>(dq), nullptr, kv_nb, kv_inds, lse2, delta, s.B, s.S,
              s.h, sl2, scale, status, 1};
  return launch_mode<D, true>(q, dout, k, v, s, pq, st);
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const void *q, const void *k, const void *v, const void *dout,
                               const Shape &s, const int32_t *kv_nb, const int32_t *kv_inds,
                               const int32_t *qt_nb, const int32_t *qt_inds, const float *lse2,
                               const float *delta, float scale, void *dq, void *dk, void *dv,
                               int *status, cudaStream_t st) {
  if (s.D == 64)
    return launch_both<64>(q, k, v, dout, s, kv_nb, kv_inds, qt_nb, qt_inds, lse2, delta, scale,
                           dq, dk, dv, status, st);
  return launch_both<128>(q, k, v, dout, s, kv_nb, kv_inds, qt_nb, qt_inds, lse2, delta, scale,
                          dq, dk, dv, status, st);
}

}  // namespace nabla
