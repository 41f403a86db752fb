// C ABI of the NABLA hot path: argument checks, workspace layout, dispatch.
// The operations and their sources are documented in include/nabla.h.
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace nabla {

namespace {

constexpr int kMaxBlocks = 2048;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_shape(int B, int S, int h, int D) {
  if (B < 1 || h < 1 || S < 64 || S % 64 != 0) return false;
  if (D != 64 && D != 128) return false;
  if (S / 64 > kMaxBlocks) return false;
  // element counts must fit the kernels' index arithmetic
  const double elems = (double)B * S * h * D;
  if (elems > 4.0e12) return false;
  if ((double)B * h * (S / 64) > 2.0e9) return false;
  return true;
}

bool valid_dtype(nabla_dtype dt) { return dt == NABLA_F32 || dt == NABLA_BF16; }

nabla_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NABLA_OK : NABLA_ERR_CUDA; }

}  // namespace

MaskWorkspace mask_workspace_layout(const Shape &s) {
  MaskWorkspace w{};
  w.mean_bytes = round_up((size_t)s.B * s.h * s.s1 * s.D * sizeof(float), 256);
  const size_t logits = (size_t)s.B * s.h * s.s1 * s.s1 * sizeof(float);
  w.qa_hi = 0;
  w.qa_lo = w.mean_bytes;
  w.ka_hi = 2 * w.mean_bytes;
  w.ka_lo = 3 * w.mean_bytes;
  w.logits = 4 * w.mean_bytes;
  w.total = round_up(w.logits + logits, 256);
  return w;
}

}  // namespace nabla

using nabla::Shape;

extern "C" {

int nabla_abi_version(void) { return 1; }

const char *nabla_status_string(nabla_status s) {
  switch (s) {
    case NABLA_OK: return "NABLA_OK";
    case NABLA_ERR_INVALID_ARG: return "NABLA_ERR_INVALID_ARG";
    case NABLA_ERR_UNSUPPORTED: return "NABLA_ERR_UNSUPPORTED";
    case NABLA_ERR_CUDA: return "NABLA_ERR_CUDA";
    case NABLA_ERR_TIMEOUT: return "NABLA_ERR_TIMEOUT";
    case NABLA_ERR_BAD_INDEX: return "NABLA_ERR_BAD_INDEX";
  }
  return "NABLA_ERR_UNKNOWN";
}

size_t nabla_build_mask_workspace_bytes(int B, int S, int h, int D) {
  if (!nabla::valid_shape(B, S, h, D)) return 0;
  return nabla::mask_workspace_layout(Shape{B, S, h, D, S / 64}).total;
}

nabla_status nabla_build_mask(const void *q, const void *k, nabla_dtype dt, int B, int S, int h,
                              int D, const uint8_t *sta, double thr, int32_t *kv_nb,
                              int32_t *kv_inds, void *workspace, size_t ws_bytes,
                              nabla_stream_t stream) {
  using namespace nabla;
  if (!valid_shape(B, S, h, D) || !valid_dtype(dt)) return NABLA_ERR_INVALID_ARG;
  if (!(thr > 0.0 && thr <= 1.0)) return NABLA_ERR_INVALID_ARG;  // also rejects NaN
  if (!q || !k || !sta || !kv_nb || !kv_inds || !workspace) return NABLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(workspace, 256) || !aligned(kv_nb, 4) ||
      !aligned(kv_inds, 4))
    return NABLA_ERR_INVALID_ARG;
  const Shape s{B, S, h, D, S / 64};
  const MaskWorkspace w = mask_workspace_layout(s);
  if (ws_bytes < w.total) return NABLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  float *qa_hi = reinterpret_cast<float *>(ws + w.qa_hi);
  float *qa_lo = reinterpret_cast<float *>(ws + w.qa_lo);
  float *ka_hi = reinterpret_cast<float *>(ws + w.ka_hi);
  float *ka_lo = reinterpret_cast<float *>(ws + w.ka_lo);
  float *L = reinterpret_cast<float *>(ws + w.logits);
  const float t = (float)(1.0 - thr);  // cut level, formed in fp64 then rounded once
  const size_t lo_off = w.mean_bytes / sizeof(float);
  cudaError_t e;
  int *status = device_status_ptr(&e);
  if (!status) return NABLA_ERR_CUDA;
  e = launch_pool(q, k, dt, s, 0, h, qa_hi, ka_hi, lo_off, st);
  if (e == cudaSuccess) e = launch_pooled_map(qa_hi, qa_lo, ka_hi, ka_lo, s, 0, h, L, status, st);
  if (e == cudaSuccess) e = launch_select(L, s, 0, h, sta, t, kv_nb, kv_inds, st);
  return from_cuda(e);
}

nabla_status nabla_build_mask_topk(const void *q, const void *k, nabla_dtype dt, int B, int S,
                                   int h, int D, double topk_ratio, int32_t *kv_nb,
                                   int32_t *kv_inds, void *workspace, size_t ws_bytes,
                                   nabla_stream_t stream) {
  using namespace nabla;
  if (!valid_shape(B, S, h, D) || !valid_dtype(dt)) return NABLA_ERR_INVALID_ARG;
  if (!(topk_ratio >= 0.0) || !std::isfinite(topk_ratio)) return NABLA_ERR_INVALID_ARG;
  if (!q || !k || !kv_nb || !kv_inds || !workspace) return NABLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(workspace, 256) || !aligned(kv_nb, 4) ||
      !aligned(kv_inds, 4))
    return NABLA_ERR_INVALID_ARG;
  const Shape s{B, S, h, D, S / 64};
  const MaskWorkspace w = mask_workspace_layout(s);
  if (ws_bytes < w.total) return NABLA_ERR_INVALID_ARG;
  // topk = min(s1, floor(ratio * s1)), the product formed in fp64
  const double prod = topk_ratio * (double)s.s1;
  const int topk = prod >= (double)s.s1 ? s.s1 : (int)std::floor(prod);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (topk == 0)
    return from_cuda(cudaMemsetAsync(kv_nb, 0, (size_t)B * h * s.s1 * sizeof(int32_t), st));
  char *ws = static_cast<char *>(workspace);
  float *qa_hi = reinterpret_cast<float *>(ws + w.qa_hi);
  float *qa_lo = reinterpret_cast<float *>(ws + w.qa_lo);
  float *ka_hi = reinterpret_cast<float *>(ws + w.ka_hi);
  float *ka_lo = reinterpret_cast<float *>(ws + w.ka_lo);
  float *L = reinterpret_cast<float *>(ws + w.logits);
  const size_t lo_off = w.mean_bytes / sizeof(float);
  cudaError_t e;
  int *status = device_status_ptr(&e);
  if (!status) return NABLA_ERR_CUDA;
  e = launch_pool(q, k, dt, s, 0, h, qa_hi, ka_hi, lo_off, st);
  if (e == cudaSuccess) e = launch_pooled_map(qa_hi, qa_lo, ka_hi, ka_lo, s, 0, h, L, status, st);
  if (e == cudaSuccess) e = launch_select_topk(L, s, 0, h, topk, kv_nb, kv_inds, st);
  return from_cuda(e);
}

static nabla_status attn_fwd_call(const void *q, const void *k, const void *v, nabla_dtype dt,
                                  int B, int S, int h, int D, const int32_t *kv_nb,
                                  const int32_t *kv_inds, float scale, void *o, float *lse,
                                  nabla_stream_t stream) {
  using namespace nabla;
  if (!valid_shape(B, S, h, D) || !valid_dtype(dt)) return NABLA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return NABLA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !kv_nb || !kv_inds) return NABLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(kv_nb, 4) || !aligned(kv_inds, 4) || !aligned(lse, 4))
    return NABLA_ERR_INVALID_ARG;
  const Shape s{B, S, h, D, S / 64};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  int *status = device_status_ptr(&e);
  if (!status) return NABLA_ERR_CUDA;
  if (dt == NABLA_BF16)
    e = launch_attn_tc(q, k, v, s, kv_nb, kv_inds, scale, o, lse, status, st);
  else
    e = launch_attn_simt(q, k, v, dt, s, kv_nb, kv_inds, scale, o, lse, status, st);
  return from_cuda(e);
}

nabla_status nabla_attn_fwd(const void *q, const void *k, const void *v, nabla_dtype dt, int B,
                            int S, int h, int D, const int32_t *kv_nb, const int32_t *kv_inds,
                            float scale, void *o, nabla_stream_t stream) {
  return attn_fwd_call(q, k, v, dt, B, S, h, D, kv_nb, kv_inds, scale, o, nullptr, stream);
}

nabla_status nabla_attn_fwd_lse(const void *q, const void *k, const void *v, nabla_dtype dt,
                                int B, int S, int h, int D, const int32_t *kv_nb,
                                const int32_t *kv_inds, float scale, void *o, float *lse,
                                nabla_stream_t stream) {
  if (!lse) return NABLA_ERR_INVALID_ARG;
  return attn_fwd_call(q, k, v, dt, B, S, h, D, kv_nb, kv_inds, scale, o, lse, stream);
}

size_t nabla_attn_bwd_workspace_bytes(int B, int S, int h, int D) {
  if (!nabla::valid_shape(B, S, h, D)) return 0;
  return nabla::bwd_workspace_layout(Shape{B, S, h, D, S / 64}).total;
}

nabla_status nabla_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dout, nabla_dtype dt, int B, int S,
                            int h, int D,
                            const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *dq,
                            void *dk, void *dv, void *workspace, size_t ws_bytes,
                            nabla_stream_t stream) {
  using namespace nabla;
  if (!valid_shape(B, S, h, D) || !valid_dtype(dt)) return NABLA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return NABLA_ERR_INVALID_ARG;
  const void *in[] = {q, k, v, o, dout};
  void *out[] = {dq, dk, dv};
  for (const void *p : in)
    if (!p || !aligned(p, 16)) return NABLA_ERR_INVALID_ARG;
  for (void *p : out)
    if (!p || !aligned(p, 16)) return NABLA_ERR_INVALID_ARG;
  if (!kv_nb || !kv_inds || !workspace || !aligned(kv_nb, 4) || !aligned(kv_inds, 4) ||
      !aligned(workspace, 256) || !aligned(lse, 16))
    return NABLA_ERR_INVALID_ARG;
  const Shape s{B, S, h, D, S / 64};
  if (ws_bytes < bwd_workspace_layout(s).total) return NABLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  int *status = device_status_ptr(&e);
  if (!status) return NABLA_ERR_CUDA;
  return from_cuda(launch_attn_bwd(q, k, v, o, lse, dout, dt, s, kv_nb, kv_inds, scale, dq, dk,
                                   dv, workspace, status, st));
}

static nabla_status fractal_call(const void *src, void *dst, bool flatten, nabla_dtype dt, int B,
                                 int T, int H, int W, int h, int D, int P,
                                 nabla_stream_t stream) {
  using namespace nabla;
  if (!valid_dtype(dt)) return NABLA_ERR_INVALID_ARG;
  if (B < 1 || T < 1 || H < 1 || W < 1 || h < 1 || D < 1 || P < 1) return NABLA_ERR_INVALID_ARG;
  if (H % P != 0 || W % P != 0) return NABLA_ERR_INVALID_ARG;
  const double tokens = (double)B * T * H * W;
  const size_t esz = dt == NABLA_BF16 ? 2 : 4;
  const size_t row_bytes = (size_t)h * D * esz;
  if (row_bytes % 16 != 0 || tokens * (double)row_bytes > 1.0e13 || tokens > 4.0e12)
    return NABLA_ERR_INVALID_ARG;
  if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16)) return NABLA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)tokens * row_bytes;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(src), b0 = reinterpret_cast<uintptr_t>(dst);
  if (a0 < b0 + bytes && b0 < a0 + bytes) return NABLA_ERR_INVALID_ARG;  // overlapping buffers
  return from_cuda(launch_fractal(src, dst, flatten, B, T, H, W, P, row_bytes,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

nabla_status nabla_fractal_flatten(const void *x, nabla_dtype dt, int B, int T, int H, int W,
                                   int h, int D, int P, void *y, nabla_stream_t stream) {
  return fractal_call(x, y, true, dt, B, T, H, W, h, D, P, stream);
}

nabla_status nabla_fractal_unflatten(const void *y, nabla_dtype dt, int B, int T, int H, int W,
                                     int h, int D, int P, void *x, nabla_stream_t stream) {
  return fractal_call(y, x, false, dt, B, T, H, W, h, D, P, stream);
}

nabla_status nabla_sta_mask(int T, int H, int W, int wt, int wh, int ww, uint8_t *sta,
                            nabla_stream_t stream) {
  if (T < 1 || H < 1 || W < 1 || wt < 0 || wh < 0 || ww < 0 || !sta) return NABLA_ERR_INVALID_ARG;
  if ((long)T * H * W > nabla::kMaxBlocks) return NABLA_ERR_INVALID_ARG;
  return nabla::from_cuda(
      nabla::launch_sta(T, H, W, wt, wh, ww, sta, reinterpret_cast<cudaStream_t>(stream)));
}

nabla_status nabla_selftest_bounded_wait(nabla_stream_t stream) {
  return nabla::from_cuda(nabla::launch_bounded_wait_probe(reinterpret_cast<cudaStream_t>(stream)));
}

nabla_status nabla_get_last_device_status(nabla_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return NABLA_ERR_CUDA;
  int *status = nabla::device_status_ptr(&e);
  if (!status) return NABLA_ERR_CUDA;
  int host = 0;
  e = cudaMemcpy(&host, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return NABLA_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    e = cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return NABLA_ERR_CUDA;
  }
  return static_cast<nabla_status>(host);
}

}  // extern "C"
