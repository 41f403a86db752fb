// K2a -- pooled map L = qa ka^T / sqrt(D) per (batch, head), on the tcgen05
// tensor cores.
//
// FastVideo API reference, page "nabla", nablaT_v2 "Map estimation": the block
// means are multiplied (qa @ ka^T) and the result divided by sqrt(D) before the
// row softmax; gist.science NABLA summary, Methodology "Reduced Attention".
//
// The cut that follows orders blocks by probability, and two blocks whose
// probabilities differ by a relative 1e-5 must still be ordered right, so the
// logits need close to fp32 accuracy; a single tf32 (or bf16) product would
// be off by ~1e-3.  Each mean is therefore split by the pool kernel into
// hi = tf32(m) and lo = tf32(m - hi), and the tile is accumulated in fp32 as
// hi*hi + hi*lo + lo*hi with kind::tf32 MMAs (the dropped lo*lo term is
// ~2^-22 of the product): three tf32 MMAs per k-step, about 1.5x the cost of
// one bf16 pass, far below the fp32 CUDA-core rate.
//
// Persistent CTAs; a work unit is a strip of 128 query blocks x all key blocks
// of one (b, h).  The strip's query means (hi and lo, 128 x D each) are loaded
// once into TMEM and serve as the A operand of every MMA of the strip; only the
// key means stream, in 32-column (128-byte swizzled) chunks of B_hi and B_lo
// through a 4-stage TMA ring, one 128-key tile after another.  Per k-step three
// kind::tf32 MMAs (lo*hi, hi*lo, hi*hi) accumulate a 128 x 128 fp32 tile in
// TMEM; two accumulators let the epilogue of one tile overlap the MMAs of the
// next.  TMEM columns: A_hi [0, 128), A_lo [128, 256), accumulators [256, 384)
// and [384, 512).  Warp roles: 0 = TMA producer, 1 = MMA issuer, 4-7 = epilogue
// (the q means already carry log2(e)/sqrt(D) -- the map is kept in base-2
// units, so the softmax that follows is a plain 2^x -- so the accumulators are
// stored as they are: 32 x 32 pieces written 128-byte-swizzled to shared memory
// and sent out by TMA stores, which also clip the ragged edges), 8-15 = strip
// loaders (hi and lo of the next strip into TMEM as soon as the MMAs of the
// current one are done, its first columns fetched ahead).  Operand
// tensors are 3-D (D, s1, B*h) so a tile never reads across a head boundary
// (out-of-range rows are zero-filled and their results are not stored).
#include <cuda.h>
#include <cstring>
#include <cudaTypedefs.h>

#include "internal.h"
#include "pdl.cuh"
#include "tc_ptx.cuh"

namespace nabla {
namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 128, kBK = 32;
constexpr int kStages = 4;
constexpr int kBBytes = kBN * kBK * 4;    // one 32-column chunk of B (16 KB)
constexpr int kStageBytes = 2 * kBBytes;  // B_hi, B_lo
constexpr int kThreads = 512;
constexpr int kEpiWarps = 4;  // one per TMEM lane quarter, four 32-column pieces each per tile
constexpr uint32_t kColAhi = 0, kColAlo = 128, kColAcc = 256;

// kind::tf32 instruction descriptor: fp32 accumulator (bits 4-5 = 1), A and B
// TF32 (format code 2 in bits 7-9 and 10-12), both K-major, N >> 3, M >> 4.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

constexpr int kStagePad = 33;  // 32 x 33 fp32 per epilogue warp: conflict-free transpose
constexpr int kPieceBytes = 32 * 32 * 4;  // one 32 x 32 fp32 output piece

struct MapSync {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], a_full, a_empty, drain;
  uint32_t tmem_slot;
  int abort;
};
// epilogue staging: two swizzled pieces per epilogue warp (TMA stores), or one
// 32 x 33 transpose tile per warp (plain stores)
constexpr int kEpiBytes = kEpiWarps * 2 * kPieceBytes;
static_assert(kEpiBytes >= kEpiWarps * 32 * kStagePad * 4, "transpose tile fits the staging area");
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + (int)sizeof(MapSync);
static_assert(kSmemBytes <= 232448, "shared memory budget");

// D[tmem] (+)= A[tmem] * B[smem desc], kind::tf32
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %4, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(accumulate), "r"(kIdesc)
      : "memory");
}

// Bulk tensor store of a shared-memory box (clipped to the tensor's bounds).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// at most one group of this thread still reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the async proxy (TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

struct MapParams {
  const float *qa_hi, *qa_lo;  // [B*h, s1, D]
  float *L;
  int h, h0, nh;  // heads per batch; this launch covers heads [h0, h0 + nh) of every batch
  int units;      // B * nh (batch, head) pairs
  int s1, D;
  int mt, nt;  // tiles along rows / columns of one head
  int *status;
};

// (batch * h + head) of the u-th (batch, head) pair of a launch.
__device__ __forceinline__ int pair_index(const MapParams &P, int u) {
  const int b = u / P.nh;
  return b * P.h + P.h0 + (u - b * P.nh);
}

// kTma: the map rows are 16-byte aligned (s1 % 4 == 0), so output pieces leave
// through TMA stores; otherwise through a shared-memory transpose and plain stores.
template <bool kTma>
__global__ void __launch_bounds__(kThreads, 1)
    pooled_map_kernel(const __grid_constant__ CUtensorMap tKh, const __grid_constant__ CUtensorMap tKl,
                      const __grid_constant__ CUtensorMap tL, MapParams P) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *epi = smem + kStages * kStageBytes;  // 1024-byte aligned
  MapSync *sync = reinterpret_cast<MapSync *>(epi + kEpiBytes);
  volatile int *abort = &sync->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long strips = (long)P.units * P.mt;
  const int chunks = P.D / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sync->full[i], 1);
      mbar_init(&sync->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sync->acc_full[i], 1);
      mbar_init(&sync->acc_empty[i], 32 * kEpiWarps);
    }
    mbar_init(&sync->a_full, 256);
    mbar_init(&sync->a_empty, 1);
    mbar_init(&sync->drain, 1);
    sync->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sync->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sync->tmem_slot;
  pdl_wait();  // the block means are written; no earlier kernel still reads L

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: B chunks of every tile of every strip
    uint32_t it = 0;
    bool ok = true;
    for (long s = blockIdx.x; s < strips && ok; s += gridDim.x) {
      const int bh = pair_index(P, (int)(s / P.mt));
      for (int nt = 0; nt < P.nt && ok; ++nt) {
        for (int c = 0; c < chunks; ++c, ++it) {
          const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
          ok = mbar_wait(&sync->empty[st], ph ^ 1u, abort, P.status, kDevTimeout);
          if (!ok) break;
          uint8_t *base = smem + st * kStageBytes;
          mbar_expect_tx(&sync->full[st], kStageBytes);
          tma_load_3d(base, &tKh, &sync->full[st], c * kBK, nt * kBN, bh);
          tma_load_3d(base + kBBytes, &tKl, &sync->full[st], c * kBK, nt * kBN, bh);
        }
      }
    }
    if (!ok) {  // let in-flight copies land before the CTA exits
      for (uint32_t e = it > (uint32_t)kStages ? it - kStages : 0u; e < it; ++e)
        mbar_wait(&sync->full[e % kStages], (e / kStages) & 1u, nullptr, P.status, kDevTimeout);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issue
    const uint64_t d0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
    uint32_t it = 0, tc = 0, ls = 0;
    bool ok = true;
    for (long s = blockIdx.x; s < strips && ok; s += gridDim.x, ++ls) {
      ok = mbar_wait(&sync->a_full, ls & 1u, abort, P.status, kDevTimeout);
      if (!ok) break;
      tc_fence_after();
      for (int nt = 0; nt < P.nt && ok; ++nt, ++tc) {
        const uint32_t ab = tc & 1u;
        ok = mbar_wait(&sync->acc_empty[ab], ((tc >> 1) & 1u) ^ 1u, abort, P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + kColAcc + ab * kBN;
        for (int c = 0; c < chunks; ++c, ++it) {
          const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
          ok = mbar_wait(&sync->full[st], ph, abort, P.status, kDevTimeout);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bhd = d0 + (uint64_t)((st * kStageBytes) >> 4);
          const uint64_t bl = bhd + (uint64_t)(kBBytes >> 4);
#pragma unroll
          for (int k8 = 0; k8 < kBK / 8; ++k8) {  // 8 tf32 = 32 B per k-step inside the atom
            const uint64_t o = (uint64_t)((k8 * 32) >> 4);
            const uint32_t col = (uint32_t)(c * kBK + k8 * 8);
            mma_tf32_ts(acc, tmem + kColAlo + col, bhd + o, (c > 0 || k8 > 0) ? 1u : 0u);
            mma_tf32_ts(acc, tmem + kColAhi + col, bl + o, 1u);
            mma_tf32_ts(acc, tmem + kColAhi + col, bhd + o, 1u);
          }
          mma_commit(&sync->empty[st]);
        }
        if (ok) mma_commit(&sync->acc_full[ab]);
      }
      if (ok) mma_commit(&sync->a_empty);  // the strip's A may be replaced once these land
    }
    mma_commit(&sync->drain);
    mbar_wait(&sync->drain, 0, nullptr, P.status, kDevTimeout);
  } else if (warp >= 8) {
    // ---- strip loaders: warps 8-11 write the hi rows, 12-15 the lo rows of the
    // next strip into TMEM (thread = TMEM lane = strip row).  The first 64
    // columns are fetched before the wait for the current strip's MMAs, so only
    // the rest of the row is on the critical path.
    const int q4 = warp & 3;
    const int part = (warp >> 2) & 1;  // 0: hi, 1: lo
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t col0 = part ? kColAlo : kColAhi;
    auto fetch = [&](const float *src, int row, int c, uint32_t (&v)[2][32]) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row < P.s1) f = *reinterpret_cast<const float4 *>(src + c + 32 * h + 4 * i);
          v[h][4 * i] = __float_as_uint(f.x);
          v[h][4 * i + 1] = __float_as_uint(f.y);
          v[h][4 * i + 2] = __float_as_uint(f.z);
          v[h][4 * i + 3] = __float_as_uint(f.w);
        }
    };
    uint32_t ls = 0;
    for (long s = blockIdx.x; s < strips && !*abort; s += gridDim.x, ++ls) {
      const int bh = pair_index(P, (int)(s / P.mt));
      const int row = (int)(s % P.mt) * kBM + r;
      const float *src = (part ? P.qa_lo : P.qa_hi) + ((size_t)bh * P.s1 + row) * P.D;
      uint32_t v[2][32];
      fetch(src, row, 0, v);  // in flight while the previous strip finishes
      if (ls > 0) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&sync->a_empty, (ls - 1) & 1u, abort,
                                                          P.status, kDevTimeout));
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st32(tmem + lane_base + col0, v[0]);
      tmem_st32(tmem + lane_base + col0 + 32, v[1]);
#pragma unroll 1
      for (int c = 64; c < P.D; c += 64) {
        fetch(src, row, c, v);
        tmem_st32(tmem + lane_base + col0 + (uint32_t)c, v[0]);
        tmem_st32(tmem + lane_base + col0 + (uint32_t)c + 32, v[1]);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sync->a_full);
    }
  } else if (warp >= 4) {
    // ---- epilogue: thread = accumulator lane = tile row; warp w owns rows
    // 32 (w % 4) .. + 31 and writes them in four 32 x 32 pieces per tile
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    uint8_t *wbuf = epi + q4 * 2 * kPieceBytes;
    float *tw = reinterpret_cast<float *>(epi) + q4 * 32 * kStagePad;
    uint32_t tc = 0, pc = 0;
    for (long s = blockIdx.x; s < strips && !*abort; s += gridDim.x) {
      const int bh = pair_index(P, (int)(s / P.mt));
      const int row0 = (int)(s % P.mt) * kBM + q4 * 32;
      for (int nt = 0; nt < P.nt; ++nt, ++tc) {
        const uint32_t ab = tc & 1u;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&sync->acc_full[ab], (tc >> 1) & 1u,
                                                          abort, P.status, kDevTimeout));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int pair = 0; pair < kBN / 64; ++pair) {
          uint32_t v[2][32];
          tmem_ld32(tmem + lane_base + kColAcc + ab * kBN + pair * 64, v[0]);
          tmem_ld32(tmem + lane_base + kColAcc + ab * kBN + pair * 64 + 32, v[1]);
          tmem_wait_ld();
          reg_fence(v[0]);
          reg_fence(v[1]);
          if (pair == kBN / 64 - 1) {  // the whole accumulator is in registers: release it
            tc_fence_before();
            mbar_arrive(&sync->acc_empty[ab]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col0 = nt * kBN + pair * 64 + h * 32;
            if (kTma) {
              // A piece wholly outside the map is neither staged nor stored: every
              // staged piece commits one bulk group, so "at most one group still
              // reading" below always means the store of the other buffer.
              if (row0 >= P.s1 || col0 >= P.s1) continue;  // uniform over the warp
              // 128-byte swizzle: 16-byte chunk k of row r sits at chunk k ^ (r & 7)
              uint8_t *buf = wbuf + (pc & 1u) * kPieceBytes;
              if (lane == 0) bulk_wait_read_1();  // the store of two pieces ago has read buf
              __syncwarp();
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4 *>(buf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                    make_uint4(v[h][4 * k], v[h][4 * k + 1], v[h][4 * k + 2], v[h][4 * k + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tL, buf, col0, row0, bh);
                bulk_commit();
              }
              ++pc;
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) tw[lane * kStagePad + i] = __uint_as_float(v[h][i]);
              __syncwarp();
              const int col = col0 + lane;
              if (col < P.s1) {
                float *out = P.L + ((size_t)bh * P.s1 + row0) * P.s1 + col;
#pragma unroll 4
                for (int rr = 0; rr < 32; ++rr)
                  if (row0 + rr < P.s1) out[(size_t)rr * P.s1] = tw[rr * kStagePad + lane];
              }
              __syncwarp();
            }
          }
        }
      }
      if (*abort) break;
    }
    if (kTma && lane == 0) bulk_wait_all();  // stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// fp32 [B*h, s1, D] viewed as (D, s1, B*h); box = 32 columns x `rows` rows x 1.
bool make_map3(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const float *ptr,
               const Shape &s, int rows) {
  cuuint64_t dims[3] = {(cuuint64_t)s.D, (cuuint64_t)s.s1, (cuuint64_t)s.B * s.h};
  cuuint64_t strides[2] = {(cuuint64_t)s.D * 4, (cuuint64_t)s.s1 * s.D * 4};
  cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 map [B*h, s1, s1] viewed as (s1 columns, s1 rows, B*h); box = 32 x 32 x 1.
bool make_map_out(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, float *ptr,
                  const Shape &s) {
  cuuint64_t dims[3] = {(cuuint64_t)s.s1, (cuuint64_t)s.s1, (cuuint64_t)s.B * s.h};
  cuuint64_t strides[2] = {(cuuint64_t)s.s1 * 4, (cuuint64_t)s.s1 * s.s1 * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_pooled_map(const float *qa_hi, const float *qa_lo, const float *ka_hi,
                              const float *ka_lo, const Shape &s, int h0, int h1, float *L,
                              int *status, cudaStream_t st) {
  cudaError_t err;
  auto enc = tensor_map_encoder(&err);
  if (!enc) return err;
  CUtensorMap tKh, tKl, tL;
  if (!make_map3(enc, &tKh, ka_hi, s, kBN) || !make_map3(enc, &tKl, ka_lo, s, kBN))
    return cudaErrorInvalidValue;
  const bool tma_out = s.s1 % 4 == 0;  // row stride a multiple of 16 bytes
  memset(&tL, 0, sizeof(tL));
  if (tma_out && !make_map_out(enc, &tL, L, s)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  auto kernel = tma_out ? pooled_map_kernel<true> : pooled_map_kernel<false>;
  if ((err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmemBytes)) != cudaSuccess)
    return err;
  MapParams p{qa_hi,
              qa_lo,
              L,
              s.h,
              h0,
              h1 - h0,
              s.B * (h1 - h0),
              s.s1,
              s.D,
              (s.s1 + kBM - 1) / kBM,
              (s.s1 + kBN - 1) / kBN,
              status};
  const long strips = (long)p.units * p.mt;
  const int grid = (int)(strips < sms ? strips : sms);
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, tKh, tKl, tL, p);
}

}  // namespace nabla
