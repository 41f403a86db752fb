// Internal launch interface between the C ABI (api.cpp) and the kernels.
// Not installed; the public contract is include/nabla.h.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "nabla.h"

namespace nabla {

struct Shape {
  int B, S, h, D, s1;
};

// Device status codes written by kernels (first writer wins); values match nabla_status.
enum : int { kDevOk = 0, kDevTimeout = NABLA_ERR_TIMEOUT, kDevBadIndex = NABLA_ERR_BAD_INDEX };

// Diagnostic: a wait nothing satisfies must end as a recorded timeout.
cudaError_t launch_bounded_wait_probe(cudaStream_t st);

// Address of the library's device status word on the current device (cached per device).
int *device_status_ptr(cudaError_t *err);

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(cudaError_t *err);

// Byte offsets of the mask-builder workspace regions (each 256-byte aligned):
// block means of q and k as tf32 hi/lo pairs, equally spaced by `mean_bytes`
// (qa_hi, qa_lo, ka_hi, ka_lo), then the fp32 pooled map.
struct MaskWorkspace {
  size_t mean_bytes, qa_hi, qa_lo, ka_hi, ka_lo, logits, total;
};
MaskWorkspace mask_workspace_layout(const Shape &s);

// The mask kernels below each cover heads [h0, h1) of every batch (the mask
// builder passes all heads).
// K1: block means of q (times log2(e)/sqrt(D)) and k -> tf32 hi at qa/ka, tf32 lo
// at +lo_off elements, each [B, h, s1, D].
cudaError_t launch_pool(const void *q, const void *k, nabla_dtype dt, const Shape &s, int h0,
                        int h1, float *qa, float *ka, size_t lo_off, cudaStream_t st);
// K2a: pooled map in base-2 units, L = qa ka^T log2(e) / sqrt(D), fp32 [B, h, s1, s1],
// on tcgen05 (3-term tf32).
cudaError_t launch_pooled_map(const float *qa_hi, const float *qa_lo, const float *ka_hi,
                              const float *ka_lo, const Shape &s, int h0, int h1, float *L,
                              int *status, cudaStream_t st);
// K2b: row softmax, ascending running-sum cut at t = 1 - thr, STA OR, CSR emit.
cudaError_t launch_select(const float *L, const Shape &s, int h0, int h1, const uint8_t *sta,
                          float t, int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st);
// K2b, top-k selector: keep the last topk blocks of each row's ascending
// (score, index) order of L (1 <= topk <= s1), listed ascending.
cudaError_t launch_select_topk(const float *L, const Shape &s, int h0, int h1, int topk,
                               int32_t *kv_nb, int32_t *kv_inds, cudaStream_t st);

// Fractal token order: whole rows of row_bytes (a multiple of 16) moved between
// [B, T, H, W, ...] raster and [B, T*H*W, ...] fractal order (flatten: raster ->
// fractal; else the inverse).
cudaError_t launch_fractal(const void *src, void *dst, bool flatten, int B, int T, int H, int W,
                           int P, size_t row_bytes, cudaStream_t st);
// K4: STA window.
cudaError_t launch_sta(int T, int H, int W, int wt, int wh, int ww, uint8_t *sta,
                       cudaStream_t st);
// K7: block-sparse attention backward.  Workspace regions (bytes, 256-aligned):
// lse2 and delta [B, h, S] fp32, the transposed CSR qt_nb [B, h, s1] and
// qt_inds [B, h, s1, s1] int32, and the word rows [B, h, s1, words] uint32.
// A bf16 o-sized scratch follows: with no caller lse, the bf16 path runs the
// tcgen05 forward once to get lse2 (its o goes there).
struct BwdWorkspace {
  size_t lse2, delta, qt_nb, qt_inds, bits, o_scratch, total;
  int words;
};
BwdWorkspace bwd_workspace_layout(const Shape &s);
cudaError_t launch_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dout, nabla_dtype dt, const Shape &s,
                            const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *dq,
                            void *dk, void *dv, void *workspace, int *status, cudaStream_t st);
// K7t: the bf16 backward's products on tcgen05 (dK, dV per key-block pair over
// the transposed lists, then dQ per query-block pair), given lse2 and delta.
cudaError_t launch_attn_bwd_tc(const void *q, const void *k, const void *v, const void *dout,
                               const Shape &s, const int32_t *kv_nb, const int32_t *kv_inds,
                               const int32_t *qt_nb, const int32_t *qt_inds, const float *lse2,
                               const float *delta, float scale, void *dq, void *dk, void *dv,
                               int *status, cudaStream_t st);
// K3: bf16 block-sparse attention on tcgen05 (lse optional).
cudaError_t launch_attn_tc(const void *q, const void *k, const void *v, const Shape &s,
                           const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *o,
                           float *lse, int *status, cudaStream_t st);
// K3f: CUDA-core block-sparse attention (fp32 storage).
cudaError_t launch_attn_simt(const void *q, const void *k, const void *v, nabla_dtype dt,
                             const Shape &s, const int32_t *kv_nb, const int32_t *kv_inds,
                             float scale, void *o, float *lse, int *status, cudaStream_t st);

}  // namespace nabla
