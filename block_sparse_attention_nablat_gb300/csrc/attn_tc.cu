// K3 -- bf16 block-sparse attention forward on the tcgen05 tensor cores.
//
// FastVideo API reference, page "nabla", NablaAttentionImpl.forward: softmax
// attention restricted to the kept 64x64 blocks of the NABLA block mask (full
// blocks, non-causal, default scale 1/sqrt(D)); gist.science NABLA summary,
// Methodology "Expansion".  The flex-attention kernel the page calls is prior
// art; this kernel is designed for sm_103a:
//
//  * Work unit = (batch, head, pair of query blocks): 128 query rows, the
//    M = 128 shape of a single-CTA tcgen05 MMA.  The unit walks the UNION of
//    the two blocks' kept-KV lists in ascending order; each entry carries two
//    membership bits, and rows of a block that did not keep an entry get P = 0
//    for it.  Blocks are paired at a stride d (block i with i + d inside each
//    run of 2d blocks), and the kernel picks d itself: before starting, every
//    CTA counts the list unions of the same fixed sample of pairs for each d
//    with 2d dividing s1 (integer counts, so all CTAs agree) and takes the d
//    with the fewest.  On a video latent the temporal neighbour (d = H*W)
//    shares more of its kept list than the horizontal one (d = 1), so fewer
//    MMAs are spent on entries only one block of the pair needs.  Persistent
//    CTAs (one per SM) take units round-robin in head-major order, so
//    co-running CTAs share one head's K/V in L2.  A unit's walk over its
//    entries starts at the key block where a sweep of s1 blocks per mean unit
//    would be after the entries its CTA has walked so far, and wraps around:
//    units of different lengths leave the CTAs at different points of their
//    lists, and this puts the CTAs of a head back in step (a head's K and V,
//    50 MB at 720p, do not stay in L2 across the staggered sweeps).  The order
//    depends on the lists alone, so results are reproducible bit for bit.
//  * A step covers two KV entries (128 keys).  Measured on this hardware, a
//    bf16 tcgen05 MMA with M = 128, K = 16 takes 48 cycles at N = 64 (two
//    thirds of the tensor rate) and N / 2 cycles from N = 128 up (the full
//    rate), so S = Q K^T is issued with N = 128 (both entries of the step in
//    one MMA, from a K "pair slot" whose rows 64..127 follow rows 0..63) and PV
//    with N = D.
//  * TMEM: O (128 x D fp32) in columns [0, 128) and three 128-column score
//    buffers.  With three buffers, QK^T of step s+2 only has to wait for the PV
//    of step s-1, which is already queued ahead of PV(s), so the tensor pipe
//    never drains between steps.
//  * Warp roles: warp 0 builds the unit's entry bitmaps from kv_inds, lists each
//    entry's two membership bits in entry order (so the softmax threads read one
//    16-bit pair per step instead of each scanning the bitmaps) and issues
//    the TMA loads of Q (once per unit) and of the K pair slots, warp 3 those of
//    the V tiles of each step into a V pair slot (two producers, so a wait for
//    a V slot never holds back the next K pair); one thread of warp 1 issues
//    every QK^T and one thread of warp 2 every PV (two issue streams, so one
//    stream's waits never leave the tensor pipe without queued work).
//  * The issuing threads, not the tensor pipe, set the step time: a step's 16
//    MMAs take 1024 cycles when issued back to back, but every mbarrier wait,
//    tcgen05.commit and fence on an issuing thread's path costs it hundreds of
//    cycles.  So each issuer waits on two barriers and commits once per step:
//    s_full, which the QK^T of step g commits, also frees K pair slot g % 3 for
//    the K loader, and pv_done, which the PV of step g commits, also frees V
//    pair slot g % 2 for the V loader.  Warps 4-7 and 8-11 are two
//    softmax groups splitting each step's columns (group x takes entry x).
//    Thread r of a group = TMEM lane r = query row r; the two threads of a row
//    exchange a flag through shared memory every step (a barrier per warp
//    pair), so both keep one bias and one O.
//  * Online softmax in base 2 with the scale folded in (packed f32x2 FMA for
//    the exponent argument).  The running maximum is only the exponent's bias:
//    each step's P is computed with the bias as it stands, and only when the
//    step's P sum exceeds 2^60 (or is infinite, for a row with no bias yet) do
//    the two threads of the row compute the row maximum, rescale O and l through
//    TMEM and redo the step.  Most steps thus need neither a row maximum nor a
//    maximum exchange, only a one-flag exchange; the result is exact either way
//    since O and l share the bias.
//  * Every mbarrier wait is bounded (1 s); on expiry the kernel records
//    NABLA_ERR_TIMEOUT, all roles stop waiting (the warp-pair barriers are
//    still met in lockstep, so no partner is left behind), in-flight MMAs and
//    copies are drained and TMEM is released.  Out-of-range or unsorted
//    kv_inds entries and out-of-range kv_nb are skipped and recorded as
//    NABLA_ERR_BAD_INDEX.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "attn_common.cuh"
#include "pdl.cuh"
#include "tc_ptx.cuh"

namespace nabla {
namespace {

using namespace tc;
using namespace tcattn;


template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;          // 64-column (128-byte) swizzle boxes
  static constexpr int kQBytes = 128 * D * 2;    // two query blocks
  static constexpr int kTileBytes = 64 * D * 2;  // one K or V block
  static constexpr int kPairBox = 128 * 128;     // one 64-column box of a K pair slot (128 rows)
  static constexpr int kPairBytes = 2 * kTileBytes;
  static constexpr int kKStages = 3;             // K pair slots (steps)
  static constexpr int kVPairs = 2;              // V pair slots (steps, two tiles each)
  static constexpr int kSBufs = 3;
  static_assert(kKStages == kSBufs, "a K pair slot is freed by its step's s_full");
  static constexpr uint32_t kSCol = 128;         // score buffer b at TMEM columns 128 + 128 b
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kIdescQK2 = idesc_bf16(128, 128, 0, 0);
  static constexpr uint32_t kIdescQK1 = idesc_bf16(128, 64, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, D, 0, 1);
  static constexpr int kThreads = 384;
  // shared-memory layout (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kPairBytes;
  static constexpr int kOffInfo = kOffV + kVPairs * kPairBytes;
  static constexpr int kOffXmax = kOffInfo + 2 * (int)sizeof(UnitInfo);  // [2 parity][2 grp][128]
  static constexpr int kOffXl = kOffXmax + 2 * 2 * 128 * 4;             // [2 grp][128]
  static constexpr int kOffXslow = kOffXl + 2 * 128 * 4;                // [2 grp][128]
  static constexpr int kOffFlags = kOffXslow + 2 * 128 * 4;             // [2 unit buffers][kMaxEntries]
  static constexpr int kOffBars = kOffFlags + 2 * kMaxEntries;
};

// All mbarriers and small shared flags, laid out by the compiler (8-byte aligned).
template <int NK, int NV, int NS>
struct SharedSync {
  uint64_t k_full[NK], v_full[NV];
  uint64_t q_full, q_empty, info_full[2], info_empty[2];
  uint64_t s_full[NS], p_full[NS], pv_done[NS];
  uint64_t o_free, drain;
  uint32_t tmem_slot;
  int abort;
};

template <int D>
using SyncOf = SharedSync<Cfg<D>::kKStages, Cfg<D>::kVPairs, Cfg<D>::kSBufs>;

template <int D>
constexpr int smem_bytes() {
  return 1024 + Cfg<D>::kOffBars + (int)sizeof(SyncOf<D>);
}
static_assert(smem_bytes<128>() <= 232448, "shared memory budget (D=128)");
static_assert(smem_bytes<64>() <= 232448, "shared memory budget (D=64)");

struct Bars {
  uint64_t *k_full, *v_full, *q_full, *q_empty, *info_full, *info_empty, *s_full, *p_full,
      *pv_done, *o_free, *drain;
};


struct Params {
  __nv_bfloat16 *o;
  float *lse;  // [B, h, S] base-2 log-sum-exp of each row's scaled scores, or null
  const int32_t *kv_nb, *kv_inds;
  int B, S, h;
  float scale_log2;
  int *status;
  int pstride;  // query blocks i and i + pstride form a pair (set in the kernel)
  int mean_union;  // mean union size of the sampled pairs (set in the kernel)
};



__device__ __forceinline__ void pair_sync(int q4) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + q4) : "memory");
}

// A softmax warp's arrival on p_full / o_free / info_empty: each lane has
// fenced its TMEM and shared-memory work before the warp sync, then lane 0
// arrives for the warp -- eight arrivals per event instead of 256 atomics on
// one barrier word, which sit on the PV issuer's critical path every step.
constexpr int kSmArrivals = 8;
__device__ __forceinline__ void sm_arrive(uint64_t *bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// P for 32 scores: 2^(s * scale_log2 - m) in fp32 (row-sum accumulators updated),
// packed to bf16 pairs in pk (16 TMEM columns' worth).
__device__ __forceinline__ void exp_pack(const uint32_t (&r)[32], uint64_t sc2, uint64_t nm2,
                                         uint64_t &acc0, uint64_t &acc1, uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float x0, x1, y0, y1;
    unf2(fma2(f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc2, nm2), x0, x1);
    unf2(fma2(f2(__uint_as_float(r[2 * i + 2]), __uint_as_float(r[2 * i + 3])), sc2, nm2), y0,
         y1);
    x0 = ex2(x0);
    x1 = ex2(x1);
    y0 = ex2(y0);
    y1 = ex2(y1);
    acc0 = add2(acc0, f2(x0, x1));
    acc1 = add2(acc1, f2(y0, y1));
    pk[i] = pack_bf16x2(x0, x1);
    pk[i + 1] = pack_bf16x2(y0, y1);
  }
}

// Row maximum of 64 scores times scale_log2 (the minimum for a negative scale).
__device__ __forceinline__ float scaled_row_max(const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                                float sl2) {
  float a0, a1, a2, a3;
  if (sl2 >= 0.f) {
    a0 = a1 = a2 = a3 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      a0 = max3(a0, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
      a1 = max3(a1, __uint_as_float(r0[i + 2]), __uint_as_float(r0[i + 3]));
      a2 = max3(a2, __uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
      a3 = max3(a3, __uint_as_float(r1[i + 2]), __uint_as_float(r1[i + 3]));
    }
    a0 = max3(a0, a1, fmaxf(a2, a3));
  } else {
    a0 = a1 = a2 = a3 = INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      a0 = min3(a0, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
      a1 = min3(a1, __uint_as_float(r0[i + 2]), __uint_as_float(r0[i + 3]));
      a2 = min3(a2, __uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
      a3 = min3(a3, __uint_as_float(r1[i + 2]), __uint_as_float(r1[i + 3]));
    }
    a0 = min3(a0, a1, fminf(a2, a3));
  }
  return a0 * sl2;
}

// A step's P is used as computed with the running maximum unless its sum exceeds
// this (then some P is huge, or the row had no maximum yet and P is infinite).
constexpr float kPBig = 1.152921504606846976e18f;  // 2^60

// On the abort path: wait (bounded, ignoring the abort flag) until the last
// copies this thread issued have landed, so none writes shared memory after exit.
template <int D>
__device__ void drain_copies(const Params &P, const Bars &bar, uint32_t gk, uint32_t kq) {
  using C = Cfg<D>;
  for (uint32_t e = gk > (uint32_t)C::kKStages ? gk - C::kKStages : 0u; e < gk; ++e)
    mbar_wait(&bar.k_full[e % C::kKStages], (e / C::kKStages) & 1u, nullptr, P.status,
              kDevTimeout);
  if (kq > 0) mbar_wait(bar.q_full, (kq - 1) & 1u, nullptr, P.status, kDevTimeout);
}

// Warp 0: entry bitmaps + TMA loads of Q (once per unit) and of the K pair slots,
// as far ahead as the K ring allows; warp 3 loads the V tiles (v_producer), so a
// wait for a V slot never holds back the next K pair.
template <int D>
__device__ void producer(const Params &P, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                         const CUtensorMap *tmV, uint8_t *smem, UnitInfo *info, const Bars &bar,
                         volatile int *abort) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  uint32_t gk = 0, kq = 0;  // K pair slots issued, Q tiles issued
  uint64_t tau = 0;         // entries walked by this CTA, plus a per-unit allowance
  bool stop = false;  // lane 0: a wait gave up; every lane leaves together at the loop top
  int k = 0;
  for (long u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    __syncwarp();
    if (__shfl_sync(0xffffffffu, (stop || *abort) ? 1 : 0, 0)) break;
    const int ub = k & 1;
    UnitInfo &inf = info[ub];
    bool ok = true;
    if (lane == 0)
      ok = mbar_wait(&bar.info_empty[ub], ((k >> 1) & 1) ^ 1, abort, P.status, kDevTimeout);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    const Unit un = decode(u, npairs, P.h);
    const long bh = (long)un.b * P.h + un.hh;
    // ---- union of the two kept lists as bitmaps
    for (int w = lane; w < kMaxWords; w += 32) {
      inf.a[w] = 0u;
      inf.b[w] = 0u;
    }
    __syncwarp();
    bool bad = false;
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const int qb = pair_block(un.pr, side, P.pstride);
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
    // The walk starts at the key block where a sweep of s1 blocks per mean unit
    // would be after the entries this CTA has walked so far (its units' lengths
    // plus a per-unit allowance), and wraps around.  CTAs walk entries at about
    // the same pace, so the CTAs on a head reach the same K/V tiles at about the
    // same time and share them in L2, while the order stays a function of the
    // lists alone (the result is reproducible bit for bit).
    const int mu = P.mean_union;
    const int start = (int)(((tau % (uint64_t)mu) * (uint64_t)s1) / (uint64_t)mu);
    // entry count, and the entries' membership bits for the softmax warps
    const int cnt = list_entries(inf, smem + C::kOffFlags + ub * kMaxEntries, lane, start);
    if (lane == 0) {
      inf.n = cnt;
      inf.start = start;
    }
    tau += (uint64_t)cnt + (cnt > 0 ? 8u : 1u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.info_full[ub]);
    if (lane != 0 || cnt == 0) continue;
    // ---- TMA loads (one thread; on failure it sets `stop` and rejoins the warp)
    if (!mbar_wait(bar.q_empty, (kq & 1) ^ 1, abort, P.status, kDevTimeout)) {
      stop = true;
      continue;
    }
    mbar_expect_tx(bar.q_full, C::kQBytes);  // a block past s1 is zero-filled
#pragma unroll
    for (int side = 0; side < 2; ++side)
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_4d(smem + C::kOffQ + c * 128 * 128 + side * 64 * 128, tmQ, bar.q_full, c * 64,
                    un.hh, pair_block(un.pr, side, P.pstride) * 64, un.b);
    ++kq;
    const int steps = (cnt + 1) >> 1;
    Cursor ck = cursor_at(inf, start);
    bool go = true;
    auto load_k = [&](int s) {  // both entries of step s into one pair slot
      // pair slot gk % 3 is free once the QK^T of step gk - 3 is done, which is
      // the completion s_full[gk % 3] signals (K slots and score buffers share
      // the step index)
      const uint32_t ks = gk % C::kKStages;
      go = go && mbar_wait(&bar.s_full[ks], ((gk / C::kKStages) & 1) ^ 1, abort, P.status,
                           kDevTimeout);
      if (!go) return;
      const int ne = (2 * s + 1 < cnt) ? 2 : 1;
      mbar_expect_tx(&bar.k_full[ks], ne * C::kTileBytes);
      uint8_t *slot = smem + C::kOffK + ks * C::kPairBytes;
      for (int x = 0; x < ne; ++x) {
        const int j = next_entry_wrap(inf, ck, start);
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_4d(slot + c * C::kPairBox + x * 64 * 128, tmK, &bar.k_full[ks], c * 64, un.hh,
                      j * 64, un.b);
      }
      ++gk;
    };
    for (int s = 0; s < steps && go; ++s) {
      load_k(s);
      if (*abort) go = false;
    }
    if (!go) stop = true;
  }
  if (lane == 0 && (stop || *abort)) drain_copies<D>(P, bar, gk, kq);
}

// Warp 3, lane 0: the V tiles of every step (its one or two entries, in entry
// order) into a V pair slot.  Pair slot g % 2 is free once the PV of step g - 2
// is done: the V loader waits on that step's pv_done, so the PV issuer spends
// one wait and one commit per step on V, not two of each.
template <int D>
__device__ void v_producer(const Params &P, const CUtensorMap *tmV, uint8_t *smem,
                           UnitInfo *info, const Bars &bar, volatile int *abort) {
  using C = Cfg<D>;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  static_assert(C::kVPairs < C::kSBufs, "pv_done of step g - kVPairs cannot have moved on");
  uint32_t gv = 0;  // steps loaded
  bool go = true;
  int k = 0;
  for (long u = blockIdx.x; u < units && go && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&bar.info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) {
      go = false;
      break;
    }
    const UnitInfo &inf = info[ub];
    const int n = inf.n;
    const Unit un = decode(u, npairs, P.h);
    const int start = inf.start;
    Cursor cv = cursor_at(inf, start);
    for (int e = 0; e < n && go; e += 2) {
      const uint32_t vp = gv % C::kVPairs;
      if (gv >= (uint32_t)C::kVPairs) {
        const uint32_t gp = gv - C::kVPairs;
        go = mbar_wait(&bar.pv_done[gp % C::kSBufs], (gp / C::kSBufs) & 1u, abort, P.status,
                       kDevTimeout);
        if (!go) break;
      }
      const int ne = e + 1 < n ? 2 : 1;
      mbar_expect_tx(&bar.v_full[vp], ne * C::kTileBytes);
      for (int x = 0; x < ne; ++x) {
        const int j = next_entry_wrap(inf, cv, start);
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_4d(smem + C::kOffV + (vp * 2 + x) * C::kTileBytes + c * 64 * 128, tmV,
                      &bar.v_full[vp], c * 64, un.hh, j * 64, un.b);
      }
      ++gv;
    }
    if (!go) break;
    mbar_arrive(&bar.info_empty[ub]);
  }
  if (!go || *abort)  // let in-flight copies land before the CTA exits
    for (uint32_t e = gv > (uint32_t)C::kVPairs ? gv - C::kVPairs : 0u; e < gv; ++e)
      mbar_wait(&bar.v_full[e % C::kVPairs], (e / C::kVPairs) & 1u, nullptr, P.status,
                kDevTimeout);
}


// Warp 1, lane 0: all QK^T MMAs.  QK^T of step g writes score buffer g % 3 once
// the PV of step g-3 (the last reader of that buffer) is done.
template <int D>
__device__ void qk_issuer(const Params &P, uint8_t *smem, UnitInfo *info, const Bars &bar,
                          uint32_t tmem, volatile int *abort) {
  using C = Cfg<D>;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  // Matrix descriptors are built once; an operand step only advances the start
  // address field (bits 0-13, address >> 4), which cannot carry for addresses
  // below 256 KB, so each MMA issues with one 64-bit add of an immediate.
  const uint64_t q_desc = smem_desc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
  const uint64_t k_desc = smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
  Ring<C::kSBufs> sb;       // score buffer of the next step; phase = its use count parity
  Ring<C::kKStages> ks;     // K pair slot of the next step
  uint32_t kq = 0;
  int k = 0;
  bool ok = true;
  for (long u = blockIdx.x; u < units && ok && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&bar.info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) break;
    const int n = info[ub].n;
    const int steps = (n + 1) >> 1;
    if (steps > 0) {
      if (!mbar_wait(bar.q_full, kq & 1, abort, P.status, kDevTimeout)) break;
      tc_fence_after();
      for (int s = 0; s < steps; ++s) {
        ok = mbar_wait(&bar.pv_done[sb.slot], sb.phase ^ 1u, abort, P.status, kDevTimeout) &&
             mbar_wait(&bar.k_full[ks.slot], ks.phase, abort, P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + C::kSCol + sb.slot * 128;
        const uint64_t kd = k_desc + (uint64_t)((ks.slot * C::kPairBytes) >> 4);
        const uint32_t idesc = (2 * s + 1 < n) ? C::kIdescQK2 : C::kIdescQK1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // 16-element k-step: 32 B inside a 128-B swizzle atom; every 4 steps the next
          // 64-column box (16 KB of Q, one 128-row box of the K pair slot)
          const uint64_t a = q_desc + (uint64_t)((((kk >> 2) * 128 * 128) + (kk & 3) * 32) >> 4);
          const uint64_t bd = kd + (uint64_t)((((kk >> 2) * C::kPairBox) + (kk & 3) * 32) >> 4);
          mma_ss(d, a, bd, idesc, kk > 0 ? 1u : 0u);
        }
        // s_full also frees K pair slot ks (= sb: both rings count steps) for the loader
        mma_commit(&bar.s_full[sb.slot]);
        if (s + 1 == steps) mma_commit(bar.q_empty);  // Q reusable after the unit's last QK^T
        sb.next();
        ks.next();
      }
      if (!ok) break;
      ++kq;
    }
    mbar_arrive(&bar.info_empty[ub]);
  }
  // never release TMEM / exit with MMAs in flight (matters only on the abort path)
  mma_commit(bar.drain);
  mbar_wait(bar.drain, 0, nullptr, P.status, kDevTimeout);
}

// Warp 2, lane 0: all PV MMAs, O += P V for each entry of a step once both softmax
// groups have written that step's P.
template <int D>
__device__ void pv_issuer(const Params &P, uint8_t *smem, UnitInfo *info, const Bars &bar,
                          uint32_t tmem, volatile int *abort) {
  using C = Cfg<D>;
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const uint64_t v_desc = smem_desc_sw128(smem_u32(smem + C::kOffV), 64 * 128, 1024);
  Ring<C::kSBufs> sb;
  Ring<C::kVPairs> vp;  // V pair slot of the next step
  uint32_t kq = 0;
  int k = 0;
  bool ok = true;
  for (long u = blockIdx.x; u < units && ok && !*abort; u += gridDim.x, ++k) {
    const int ub = k & 1;
    if (!mbar_wait(&bar.info_full[ub], (k >> 1) & 1, abort, P.status, kDevTimeout)) break;
    const int n = info[ub].n;
    const int steps = (n + 1) >> 1;
    if (steps > 0) {
      // O of the previous unit must have been read out before the first PV overwrites it
      if (kq > 0 && !mbar_wait(bar.o_free, (kq - 1) & 1u, abort, P.status, kDevTimeout)) break;
      for (int s = 0; s < steps; ++s) {
        ok = mbar_wait(&bar.p_full[sb.slot], sb.phase, abort, P.status, kDevTimeout) &&
             mbar_wait(&bar.v_full[vp.slot], vp.phase, abort, P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        for (int x = 0; x < 2 && 2 * s + x < n; ++x) {
          const uint64_t vd = v_desc + (uint64_t)(((vp.slot * 2 + x) * C::kTileBytes) >> 4);
          const uint32_t a0 = tmem + C::kSCol + sb.slot * 128 + x * 64;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem, a0 + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), C::kIdescPV,
                   (s > 0 || x > 0 || kk > 0) ? 1u : 0u);  // next 16 KV rows
        }
        // frees score buffer sb for QK^T and V pair slot vp for the V loader
        mma_commit(&bar.pv_done[sb.slot]);
        sb.next();
        vp.next();
      }
      if (!ok) break;
      ++kq;
    }
    mbar_arrive(&bar.info_empty[ub]);
  }
  mma_commit(bar.drain);
  mbar_wait(bar.drain, 0, nullptr, P.status, kDevTimeout);
}

// Warps 4-11: two softmax groups splitting each step's columns + the epilogue.
template <int D>
__device__ void softmax_epilogue(const Params &P, UnitInfo *info, uint8_t *smem, const Bars &bar,
                                 uint32_t tmem, volatile int *abort) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = (warp - 4) >> 2;  // takes entry grp of every step; owns O columns grp*D/2..
  const int q4 = warp & 3;          // TMEM lane quadrant; partner warp = same q4, other group
  const int row = q4 * 32 + lane;
  const int half = row >> 6;
  const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
  float *xmax = reinterpret_cast<float *>(smem + C::kOffXmax);
  float *xl = reinterpret_cast<float *>(smem + C::kOffXl);
  float *xslow = reinterpret_cast<float *>(smem + C::kOffXslow);
  const int s1 = P.S >> 6, npairs = (s1 + 1) >> 1;
  const long units = (long)P.B * P.h * npairs;
  const float sl2 = P.scale_log2;
  uint32_t gs = 0;
  int k = 0;
  bool live = true;  // false after a wait gave up: keep meeting the pair barriers, do no work
  for (long u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    const int ub = k & 1;
    live = __all_sync(0xffffffffu, live && mbar_wait(&bar.info_full[ub], (k >> 1) & 1, abort,
                                                      P.status, kDevTimeout));
    // both threads of a row must run the same number of pair barriers: agree on `live`
    // (and so on n) through the pair exchange slot
    xl[grp * 128 + row] = live ? 1.f : 0.f;
    pair_sync(q4);
    live = __all_sync(0xffffffffu, live && xl[(grp ^ 1) * 128 + row] != 0.f);
    pair_sync(q4);
    const int n = live ? info[ub].n : 0;
    const int steps = (n + 1) >> 1;
    const Unit un = decode(u, npairs, P.h);
    const int qb = pair_block(un.pr, half, P.pstride);
    float m_run = -INFINITY, l_run = 0.f;
    // the two entries' membership bits of step s, one byte each, listed by the
    // producer (one 16-bit load per step instead of a bitmap scan per thread)
    const uint16_t *fl = reinterpret_cast<const uint16_t *>(smem + C::kOffFlags + ub * kMaxEntries);
    for (int s = 0; s < steps; ++s) {
      const uint32_t g = gs + s, b = g % C::kSBufs, use = g / C::kSBufs;
      const bool has1 = 2 * s + 1 < n;
      const uint32_t pr = fl[s];
      const uint32_t f0 = pr & 0xffu, f1 = has1 ? pr >> 8 : 0u;
      const bool mine = grp == 0 || has1;
      const bool act = mine && ((((grp ? f1 : f0) >> half) & 1u) != 0u);
      live = __all_sync(0xffffffffu, live && mbar_wait(&bar.s_full[b], use & 1u, abort, P.status,
                                                        kDevTimeout));
      tc_fence_after();
      const uint32_t sbase = tmem + lane_base + C::kSCol + b * 128 + grp * 64;
      uint32_t r0[32], r1[32];
      if (live && act) {
        tmem_ld32(sbase, r0);
        tmem_ld32(sbase + 32, r1);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
      }
      // P with the running maximum as it stands.  The maximum only serves as the
      // exponent's bias, and the result is exact for any bias that keeps P finite,
      // so it is raised only when this step's P would be huge (or infinite: a row
      // with no maximum yet).  The two threads of a row agree on that through the
      // exchange slot, and only then compute the row maximum, rescale O and l,
      // and redo the step's P.
      uint32_t pk0[16], pk1[16];
      float ssum = 0.f;
      auto step_p = [&]() {
        const uint64_t sc2 = f2(sl2, sl2), nm2 = f2(-m_run, -m_run);
        uint64_t acc0 = f2(0.f, 0.f), acc1 = acc0;
        exp_pack(r0, sc2, nm2, acc0, acc1, pk0);
        exp_pack(r1, sc2, nm2, acc0, acc1, pk1);
        float s0, s1v, s2, s3;
        unf2(acc0, s0, s1v);
        unf2(acc1, s2, s3);
        ssum = (s0 + s1v) + (s2 + s3);
      };
      if (live && act) step_p();
      const bool big = !(ssum <= kPBig);  // also for an infinite or NaN sum
      float *xm = xmax + (size_t)(g & 1u) * 2 * 128;
      xm[grp * 128 + row] = big ? 1.f : 0.f;
      pair_sync(q4);
      const bool need = big || xm[(grp ^ 1) * 128 + row] != 0.f;
      if (__any_sync(0xffffffffu, need)) {
        const float mx = (need && live && act) ? scaled_row_max(r0, r1, sl2) : -INFINITY;
        xslow[grp * 128 + row] = mx;
        pair_sync(q4);
        const float m_new = need ? fmaxf(m_run, fmaxf(mx, xslow[(grp ^ 1) * 128 + row])) : m_run;
        const bool resc = need && m_run != -INFINITY && m_new > m_run;
        if (__any_sync(0xffffffffu, resc)) {
          // O must hold every PV up to the previous step before it is rescaled;
          // each group rescales its half of the D columns (the decision is the same
          // in both groups, both hold the same m_run)
          const uint32_t gp = g - 1;
          const float alpha = resc ? ex2(m_run - m_new) : 1.0f;
          live = __all_sync(0xffffffffu,
                            live && mbar_wait(&bar.pv_done[gp % C::kSBufs], (gp / C::kSBufs) & 1u,
                                              abort, P.status, kDevTimeout));
          if (live) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              const uint32_t ta = tmem + lane_base + grp * (D / 2) + c * 16;
              uint32_t t[16];
              tmem_ld16(ta, t);
              tmem_wait_ld();
              reg_fence16(t);
#pragma unroll
              for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
              tmem_st16(ta, t);
            }
            tmem_wait_st();
          }
          if (resc) l_run *= alpha;
        }
        if (need) m_run = m_new;
        if (need && live && act) step_p();
      }
      if (live && mine) {
        if (act) {
          tmem_st16(sbase, pk0);
          tmem_st16(sbase + 16, pk1);
          l_run += ssum;
        } else {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
          tmem_st16(sbase, pk);
          tmem_st16(sbase + 16, pk);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      sm_arrive(&bar.p_full[b], lane);
    }
    // ---- epilogue: O / (l_0 + l_1) -> bf16; each group writes its half of the columns
    if (steps > 0) {
      const uint32_t gl = gs + steps - 1;
      live = __all_sync(0xffffffffu,
                        live && mbar_wait(&bar.pv_done[gl % C::kSBufs], (gl / C::kSBufs) & 1u,
                                          abort, P.status, kDevTimeout));
      tc_fence_after();
    }
    xl[grp * 128 + row] = live ? l_run : -1.f;  // l >= 0; -1 marks a half that gave up
    pair_sync(q4);
    const float l_other = xl[(grp ^ 1) * 128 + row];
    pair_sync(q4);  // both read before the slot is written again
    live = __all_sync(0xffffffffu, live && l_other >= 0.f);
    const float lt = l_run + l_other;
    const float inv = lt > 0.f ? 1.0f / lt : 0.f;
    const bool row_valid = qb < s1;
    if (P.lse && grp == 0 && live && row_valid)
      P.lse[((size_t)un.b * P.h + un.hh) * P.S + (size_t)qb * 64 + (row & 63)] =
          lt > 0.f ? m_run + log2f(lt) : -INFINITY;
    __nv_bfloat16 *orow =
        P.o + (((size_t)un.b * P.S + (size_t)qb * 64 + (row & 63)) * P.h + un.hh) * D;
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      const int c = grp * (D / 32) + cc;  // this group's 16-column pieces
      uint32_t t[16];
      if (live && steps > 0) {
        tmem_ld16(tmem + lane_base + c * 16, t);
        tmem_wait_ld();
        reg_fence16(t);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = 0u;
      }
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = pack_bf16x2(__uint_as_float(t[2 * i]) * inv, __uint_as_float(t[2 * i + 1]) * inv);
      if (live && row_valid) {
        // streaming stores: o is not read again here, so its lines should not
        // linger dirty in L2 for the next kernel to write back
        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
        __stcs(dst, make_uint4(w[0], w[1], w[2], w[3]));
        __stcs(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
      }
    }
    tc_fence_before();
    if (steps > 0) sm_arrive(bar.o_free, lane);
    sm_arrive(&bar.info_empty[ub], lane);
    gs += steps;
    if (!live) break;  // both halves of every pair leave at the same unit
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, Params P) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  UnitInfo *info = reinterpret_cast<UnitInfo *>(smem + C::kOffInfo);
  SyncOf<D> *sync = reinterpret_cast<SyncOf<D> *>(smem + C::kOffBars);
  Bars bar;
  bar.k_full = sync->k_full;
  bar.v_full = sync->v_full;
  bar.q_full = &sync->q_full;
  bar.q_empty = &sync->q_empty;
  bar.info_full = sync->info_full;
  bar.info_empty = sync->info_empty;
  bar.s_full = sync->s_full;
  bar.p_full = sync->p_full;
  bar.pv_done = sync->pv_done;
  bar.o_free = &sync->o_free;
  bar.drain = &sync->drain;
  uint32_t *tmem_slot = &sync->tmem_slot;
  volatile int *abort = &sync->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kKStages; ++i) mbar_init(&bar.k_full[i], 1);
    for (int i = 0; i < C::kVPairs; ++i) mbar_init(&bar.v_full[i], 1);
    mbar_init(bar.q_full, 1);
    mbar_init(bar.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.info_full[i], 1);
      mbar_init(&bar.info_empty[i], kSmArrivals + 3);  // softmax warps, both MMA issuers, V loader
    }
    for (int i = 0; i < C::kSBufs; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.p_full[i], kSmArrivals);
      mbar_init(&bar.pv_done[i], 1);
    }
    mbar_init(bar.o_free, kSmArrivals);
    mbar_init(bar.drain, 2);  // one commit per MMA-issuing thread
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
  pdl_wait();  // kv_nb / kv_inds and q, k, v are written; no earlier kernel still reads o
  // the K / V staging area is free until the producer starts
  static_assert(sizeof(StrideScratch) <= (size_t)C::kOffInfo - C::kOffK, "stride scratch fits");
  Params Pp = P;
  Pp.pstride = choose_pair_stride(P, reinterpret_cast<StrideScratch *>(smem + C::kOffK),
                                  &Pp.mean_union);

  if (warp == 0) {
    producer<D>(Pp, &tmQ, &tmK, &tmV, smem, info, bar, abort);
  } else if (warp == 1) {
    if (lane == 0) qk_issuer<D>(Pp, smem, info, bar, tmem, abort);
    __syncwarp();
  } else if (warp == 2) {
    if (lane == 0) pv_issuer<D>(Pp, smem, info, bar, tmem, abort);
    __syncwarp();
  } else if (warp == 3) {
    if (lane == 0) v_producer<D>(Pp, &tmV, smem, info, bar, abort);
    __syncwarp();
  } else if (warp >= 4) {
    softmax_epilogue<D>(Pp, info, smem, bar, tmem, abort);
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

template <int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, const Shape &s,
                     const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                     float *lse, int *status, cudaStream_t st) {
  using C = Cfg<D>;
  cudaError_t err;
  auto enc = tensor_map_encoder(&err);
  if (!enc) return err;
  CUtensorMap mq, mk, mv;
  if (!make_map(enc, &mq, q, s, 64) || !make_map(enc, &mk, k, s, 64) ||
      !make_map(enc, &mv, v, s, 64))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  auto kern = attn_tc_kernel<D>;
  if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem_bytes<D>())) != cudaSuccess)
    return err;
  const long units = (long)s.B * s.h * ((s.s1 + 1) / 2);
  const int grid = (int)(units < sms ? units : sms);
  Params p{static_cast<__nv_bfloat16 *>(o), lse, kv_nb, kv_inds, s.B, s.S, s.h,
           scale * 1.4426950408889634f, status, 1};
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), smem_bytes<D>(), st, mq, mk, mv, p);
}

}  // namespace

cudaError_t launch_attn_tc(const void *q, const void *k, const void *v, const Shape &s,
                           const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                           float *lse, int *status, cudaStream_t st) {
  if (s.D == 64) return launch_d<64>(q, k, v, s, kv_nb, kv_inds, scale, o, lse, status, st);
  return launch_d<128>(q, k, v, s, kv_nb, kv_inds, scale, o, lse, status, st);
}

}  // namespace nabla
