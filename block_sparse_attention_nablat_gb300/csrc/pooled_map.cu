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
// Persistent CTAs; tile = 128 query blocks x 256 key blocks of one (b, h);
// K = D streamed in 32-column (128-byte swizzled) chunks of the four operands
// through a 2-stage TMA ring; the accumulator lives in TMEM (two 256-column
// buffers, so the epilogue of one tile overlaps the MMAs of the next); the
// epilogue scales by log2(e)/sqrt(D) -- the map is kept in base-2 units, so
// the softmax that follows is a plain 2^x -- and writes fp32 rows, transposed
// through shared memory into 128-byte row segments.  Operand
// tensors are 3-D (D, s1, B*h) so a tile never reads across a head boundary
// (out-of-range rows are zero-filled and their results are not stored).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace nabla {
namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 256, kBK = 32;
constexpr int kStages = 2;
constexpr int kABytes = kBM * kBK * 4;  // one operand chunk of A (16 KB)
constexpr int kBBytes = kBN * kBK * 4;  // one operand chunk of B (32 KB)
constexpr int kStageBytes = 2 * kABytes + 2 * kBBytes;  // A_hi, A_lo, B_hi, B_lo
constexpr int kThreads = 256;

// kind::tf32 instruction descriptor: fp32 accumulator (bits 4-5 = 1), A and B
// TF32 (format code 2 in bits 7-9 and 10-12), both K-major, N >> 3, M >> 4.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

constexpr int kStagePad = 33;  // 32 x 33 fp32 per epilogue warp: conflict-free transpose

struct MapSync {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_slot;
  int abort;
};
constexpr int kTransBytes = 4 * 32 * kStagePad * 4;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kTransBytes + (int)sizeof(MapSync);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %4, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(kIdesc)
      : "memory");
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
  float *L;
  int h, h0, nh;  // heads per batch; this launch covers heads [h0, h0 + nh) of every batch
  int units;      // B * nh (batch, head) pairs
  int s1, D;
  int mt, nt;  // tiles along rows / columns of one head
  float scale;
  int *status;
};

// (batch * h + head) of the u-th (batch, head) pair of a launch.
__device__ __forceinline__ int pair_index(const MapParams &P, int u) {
  const int b = u / P.nh;
  return b * P.h + P.h0 + (u - b * P.nh);
}

__global__ void __launch_bounds__(kThreads, 1)
    pooled_map_kernel(const __grid_constant__ CUtensorMap tQh, const __grid_constant__ CUtensorMap tQl,
                      const __grid_constant__ CUtensorMap tKh, const __grid_constant__ CUtensorMap tKl,
                      MapParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float *trans = reinterpret_cast<float *>(smem + kStages * kStageBytes);
  MapSync *sync = reinterpret_cast<MapSync *>(smem + kStages * kStageBytes + kTransBytes);
  volatile int *abort = &sync->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long tiles = (long)P.units * P.mt * P.nt;
  const int chunks = P.D / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sync->full[i], 1);
      mbar_init(&sync->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sync->acc_full[i], 1);
      mbar_init(&sync->acc_empty[i], 128);
    }
    mbar_init(&sync->drain, 1);
    sync->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sync->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sync->tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    uint32_t it = 0;
    for (long t = blockIdx.x; t < tiles && !*abort; t += gridDim.x) {
      const int u = (int)(t / (P.mt * P.nt));
      const int rem = (int)(t - (long)u * P.mt * P.nt);
      const int bh = pair_index(P, u);
      const int m0 = (rem / P.nt) * kBM, n0 = (rem % P.nt) * kBN;
      for (int c = 0; c < chunks; ++c, ++it) {
        const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
        if (!mbar_wait(&sync->empty[st], ph ^ 1u, abort, P.status, kDevTimeout)) break;
        uint8_t *base = smem + st * kStageBytes;
        mbar_expect_tx(&sync->full[st], kStageBytes);
        tma_load_3d(base, &tQh, &sync->full[st], c * kBK, m0, bh);
        tma_load_3d(base + kABytes, &tQl, &sync->full[st], c * kBK, m0, bh);
        tma_load_3d(base + 2 * kABytes, &tKh, &sync->full[st], c * kBK, n0, bh);
        tma_load_3d(base + 2 * kABytes + kBBytes, &tKl, &sync->full[st], c * kBK, n0, bh);
      }
    }
    if (*abort) {  // let in-flight copies land before the CTA exits
      for (uint32_t e = it > (uint32_t)kStages ? it - kStages : 0u; e < it; ++e)
        mbar_wait(&sync->full[e % kStages], (e / kStages) & 1u, nullptr, P.status, kDevTimeout);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issue
    const uint64_t d0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (long t = blockIdx.x; t < tiles && ok && !*abort; t += gridDim.x, ++tc) {
      const uint32_t ab = tc & 1u;
      ok = mbar_wait(&sync->acc_empty[ab], ((tc >> 1) & 1u) ^ 1u, abort, P.status, kDevTimeout);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = tmem + ab * 256;
      for (int c = 0; c < chunks; ++c, ++it) {
        const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
        ok = mbar_wait(&sync->full[st], ph, abort, P.status, kDevTimeout);
        if (!ok) break;
        tc_fence_after();
        const uint64_t ah = d0 + (uint64_t)((st * kStageBytes) >> 4);
        const uint64_t al = ah + (uint64_t)(kABytes >> 4);
        const uint64_t bhd = ah + (uint64_t)((2 * kABytes) >> 4);
        const uint64_t bl = bhd + (uint64_t)(kBBytes >> 4);
#pragma unroll
        for (int k8 = 0; k8 < kBK / 8; ++k8) {  // 8 tf32 = 32 B per k-step inside the atom
          const uint64_t o = (uint64_t)((k8 * 32) >> 4);
          mma_tf32(acc, al + o, bhd + o, (c > 0 || k8 > 0) ? 1u : 0u);
          mma_tf32(acc, ah + o, bl + o, 1u);
          mma_tf32(acc, ah + o, bhd + o, 1u);
        }
        mma_commit(&sync->empty[st]);
      }
      if (!ok) break;
      mma_commit(&sync->acc_full[ab]);
    }
    mma_commit(&sync->drain);
    mbar_wait(&sync->drain, 0, nullptr, P.status, kDevTimeout);
  } else if (warp >= 4) {
    // ---- epilogue: thread = accumulator lane = tile row.  Each warp owns 32 rows;
    // every 32-column piece is transposed through shared memory so that each
    // store instruction writes one contiguous 128-byte segment of one row.
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    float *tw = trans + q4 * 32 * kStagePad;
    uint32_t tc = 0;
    for (long t = blockIdx.x; t < tiles && !*abort; t += gridDim.x, ++tc) {
      const uint32_t ab = tc & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&sync->acc_full[ab], (tc >> 1) & 1u, abort,
                                                        P.status, kDevTimeout));
      if (!ok) break;
      tc_fence_after();
      const int u = (int)(t / (P.mt * P.nt));
      const int rem = (int)(t - (long)u * P.mt * P.nt);
      const int bh = pair_index(P, u);
      const int row0 = (rem / P.nt) * kBM + q4 * 32, n0 = (rem % P.nt) * kBN;
      (void)r;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + ab * 256 + c * 32, v);
        tmem_wait_ld();
        reg_fence(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) tw[lane * kStagePad + i] = __uint_as_float(v[i]) * P.scale;
        __syncwarp();
        const int col = n0 + c * 32 + lane;
        if (col < P.s1) {
          float *out = P.L + ((size_t)bh * P.s1 + row0) * P.s1 + col;
#pragma unroll 4
          for (int rr = 0; rr < 32; ++rr)
            if (row0 + rr < P.s1) out[(size_t)rr * P.s1] = tw[rr * kStagePad + lane];
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(&sync->acc_empty[ab]);
    }
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

}  // namespace

cudaError_t launch_pooled_map(const float *qa_hi, const float *qa_lo, const float *ka_hi,
                              const float *ka_lo, const Shape &s, int h0, int h1, float *L,
                              int *status, cudaStream_t st) {
  cudaError_t err;
  auto enc = tensor_map_encoder(&err);
  if (!enc) return err;
  CUtensorMap tQh, tQl, tKh, tKl;
  if (!make_map3(enc, &tQh, qa_hi, s, kBM) || !make_map3(enc, &tQl, qa_lo, s, kBM) ||
      !make_map3(enc, &tKh, ka_hi, s, kBN) || !make_map3(enc, &tKl, ka_lo, s, kBN))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  if ((err = cudaFuncSetAttribute(pooled_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmemBytes)) != cudaSuccess)
    return err;
  MapParams p{L,
              s.h,
              h0,
              h1 - h0,
              s.B * (h1 - h0),
              s.s1,
              s.D,
              (s.s1 + kBM - 1) / kBM,
              (s.s1 + kBN - 1) / kBN,
              (float)(1.4426950408889634 / sqrt((double)s.D)),
              status};
  const long tiles = (long)p.units * p.mt * p.nt;
  const int grid = (int)(tiles < sms ? tiles : sms);
  pooled_map_kernel<<<grid, kThreads, kSmemBytes, st>>>(tQh, tQl, tKh, tKl, p);
  return cudaGetLastError();
}

}  // namespace nabla
