/*
 * nabla.h -- C ABI of the GB300 (sm_103a) NABLA hot path.
 *
 * NABLA (Neighborhood-Adaptive Block-Level Attention) builds a data-dependent
 * 64x64 block mask from mean-pooled queries and keys and then runs softmax
 * attention over the kept blocks only.  Sources restated here:
 *   [P1] FastVideo API reference, page "nabla": nablaT_v2 ("Map estimation",
 *        "Map binarization", BlockMask creation), NablaAttentionImpl.forward,
 *        NablaAttentionMetadata.
 *   [P4] gist.science technical summary of "NABLA: Neighborhood Adaptive
 *        Block-Level Attention", Methodology.
 *
 * Conventions shared by every entry point:
 *   - q, k, v, o are dense, C-contiguous [B, S, h, D] tensors ([P1] forward:
 *     "q/k/v: [B, S, heads, head_dim]"), element type given by nabla_dtype.
 *     S must be a multiple of 64 and S/64 (= s1, the number of blocks) at most
 *     2048; D is 64 or 128.
 *   - Every pointer argument is DEVICE memory owned by the caller.  q, k, v, o
 *     must be 16-byte aligned, the workspace 256-byte aligned, kv_nb and kv_inds
 *     4-byte aligned; sta has no alignment rule.  The library allocates no device memory
 *     and keeps no state between calls other than a device status word (see
 *     nabla_get_last_device_status) and the statically reserved scratch array
 *     of nabla_build_mask_noalloc.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) of the CURRENT device.  A returned NABLA_OK means
 *     the arguments were valid and the kernels were launched.
 *   - The mask and attention kernels are launched with programmatic dependent
 *     launch: each lets the next kernel of the stream start its prologue early
 *     and waits for the previous kernel to complete before it touches device
 *     memory, so stream order is kept whatever precedes the call.  Setting
 *     NABLA_DISABLE_PDL=1 in the environment (read once per process) gives
 *     plain launches.
 *   - Errors are returned, never raised on the device: invalid arguments are
 *     rejected on the host before anything is launched; launch failures give
 *     NABLA_ERR_CUDA; device-side conditions (a bounded wait that gave up, an
 *     out-of-range block index) are recorded in a device status word and
 *     reported by nabla_get_last_device_status.
 *   - Causal masking is not offered ([P1] NablaAttentionImpl rejects causal).
 *     There is no sequence-parallel entry point: the mask spans the whole
 *     sequence ([P1] module description).
 */
#ifndef NABLA_H
#define NABLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st *nabla_stream_t;

typedef enum {
  NABLA_OK = 0,
  NABLA_ERR_INVALID_ARG = 1, /* bad shape, dtype, threshold, pointer or size */
  NABLA_ERR_UNSUPPORTED = 2, /* valid request this library cannot serve (e.g. no sm_103 device) */
  NABLA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  NABLA_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
  NABLA_ERR_BAD_INDEX = 5    /* kv_nb / kv_inds held an out-of-range entry (skipped) */
} nabla_status;

typedef enum {
  NABLA_F32 = 0, /* float32 storage, float32 arithmetic */
  NABLA_BF16 = 1 /* bfloat16 storage, float32 accumulation */
} nabla_dtype;

/* Version of this ABI (bumped on any signature change). */
int nabla_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *nabla_status_string(nabla_status s);

/*
 * Scratch bytes nabla_build_mask needs for a shape: the block means of q and k
 * as tf32 hi/lo pairs (four fp32 [B, h, s1, D] arrays) and the fp32 pooled map
 * ([B, h, s1, s1]), each region 256-byte aligned.  Returns 0 for an invalid
 * shape.
 *
 * After a nabla_build_mask call the workspace holds, for inspection (M =
 * B*h*s1*D*4 rounded up to a multiple of 256 bytes):
 *   [0, M)         hi parts of the query means times log2(e)/sqrt(D),
 *   [M, 2M)        their lo parts,
 *   [2M, 3M)       hi parts of the key means,   [3M, 4M) their lo parts,
 *   [4M, 4M + B*h*s1*s1*4)  the pooled map in base-2 units,
 *                  L[b,h,i,j] = <qa_i, ka_j> log2(e) / sqrt(D), fp32.
 * Any bytes after these are private to the library.
 */
size_t nabla_build_mask_workspace_bytes(int B, int S, int h, int D);

/*
 * nabla_build_mask -- the nablaT_v2 mask builder ([P1] nablaT_v2; [P4]
 * Downsampling, Reduced Attention, CDF Thresholding, Hybrid Integration).
 *
 * For every (b, h, query block i):
 *   qa_i = mean of the 64 query tokens of block i, ka_j likewise for keys;
 *   p_i  = softmax_j( <qa_i, ka_j> / sqrt(D) );
 *   sort p_i ascending (ties: lower block index first), running sum c;
 *   block j is kept iff c(j) >= 1 - thr, or sta[i*s1 + j] != 0;
 *   kv_nb[(b*h + hh)*s1 + i]           = number of kept blocks,
 *   kv_inds[((b*h + hh)*s1 + i)*s1 + n] = n-th kept block, ascending, n < kv_nb.
 * Entries of a kv_inds row at positions >= kv_nb are left unwritten.
 *
 *   q, k       [B, S, h, D] device, element type dt.
 *   sta        [s1, s1] device uint8, 0/1, shared by every batch and head
 *              ([P1] NablaAttentionMetadata: a block-level [1,1,S/64,S/64] window).
 *   thr        kept-mass threshold, 0 < thr <= 1 (thr = 1 keeps every block).
 *   kv_nb      [B, h, s1] device int32, written.
 *   kv_inds    [B, h, s1, s1] device int32, written (kept prefix of each row).
 *   workspace  device scratch of ws_bytes >= nabla_build_mask_workspace_bytes().
 * Arithmetic is fp32 (means accumulated in fp32 from the stored values); the
 * result can differ from an exact evaluation only for blocks whose running
 * sum lies within float32 rounding of 1 - thr.
 * Errors: NABLA_ERR_INVALID_ARG for S % 64 != 0, s1 > 2048, D not in {64,128},
 * B or h < 1, thr outside (0, 1], NULL or misaligned pointers, short workspace.
 */
nabla_status nabla_build_mask(const void *q, const void *k, nabla_dtype dt, int B, int S,
                              int h, int D, const uint8_t *sta, double thr, int32_t *kv_nb,
                              int32_t *kv_inds, void *workspace, size_t ws_bytes,
                              nabla_stream_t stream);

/*
 * nabla_build_mask_noalloc -- nabla_build_mask for callers that cannot
 * allocate device memory.  The NABLA pages have no counterpart; this entry
 * point is a property of this library only.
 *
 * Some callers cannot call cudaMalloc: an engine that reserves all device
 * memory for its own pool at start-up and forbids allocation afterwards, a
 * latency-critical loop that cannot afford the device-wide synchronisation
 * cudaMalloc and cudaFree may imply, or a plug-in running inside a host
 * program whose memory budget it does not control.  This variant needs no
 * workspace argument: its scratch (the fp32 block means and pooled map) is a
 * NABLA_NOALLOC_SCRATCH_BYTES array the library defines in device memory.
 * Every GPU that loads the library holds that array until the process exits.
 *
 * Arguments, result and errors are those of nabla_build_mask, minus the
 * workspace, and the result is identical, plus:
 *   - shapes whose nabla_build_mask_workspace_bytes() exceeds
 *     NABLA_NOALLOC_SCRATCH_BYTES are rejected with NABLA_ERR_UNSUPPORTED
 *     before anything is launched;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current) and keeps it for the
 *     process; make that first call before any stream capture.  First calls
 *     from several host threads are safe (the lookup is serialised).  A
 *     cudaDeviceReset unloads the library's device code and makes the kept
 *     address stale: do not call this entry point on that device again in
 *     the same process after a reset;
 *   - all calls share the one array, which keeps the last call's contents;
 *     the kernels overwrite every scratch element they read, so nothing needs
 *     clearing, but calls whose kernels overlap on the GPU (different streams,
 *     or unordered host threads) race on it and must be serialised;
 *   - it calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define NABLA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
nabla_status nabla_build_mask_noalloc(const void *q, const void *k, nabla_dtype dt, int B, int S,
                                      int h, int D, const uint8_t *sta, double thr,
                                      int32_t *kv_nb, int32_t *kv_inds, nabla_stream_t stream);

/*
 * nabla_build_mask_topk -- the top-k block selector (FastVideo API reference,
 * attention backends index, sla.get_block_map), run on the same block means
 * and pooled map as nabla_build_mask.
 *
 * For every (b, h, query block i), with qa_i the mean of the 64 query tokens
 * of block i and kc_j the mean of the 64 keys of block j after smooth-k (k
 * minus its mean over the sequence, per batch, head and channel):
 *   score_ij = <qa_i, kc_j>;  topk = min(s1, floor(topk_ratio * s1));
 *   the topk blocks j of largest score_ij are kept (equal scores: the higher
 *   block index ranks higher, i.e. the kept set is the last topk of the
 *   ascending (score, index) order);
 *   kv_nb / kv_inds as for nabla_build_mask (every row holds topk blocks,
 *   listed ascending; the page's sparse_map is the row's indicator).
 * Smooth-k subtracts <qa_i, mean k> from the whole of row i, and the pooled
 * map's 1/sqrt(D) scale is positive, so neither changes a row's order: the
 * library ranks the rows of the fp32 pooled map <qa_i, ka_j> / sqrt(D) that
 * nabla_build_mask computes.  The result can differ from an exact evaluation
 * only where two scores of a row lie within float32 rounding of each other at
 * the topk-th place.  No STA window is applied (the page has none).
 *
 *   q, k        [B, S, h, D] device, element type dt.
 *   topk_ratio  finite, >= 0; topk = 0 writes kv_nb = 0 and no kv_inds.
 *   kv_nb, kv_inds, workspace, ws_bytes: as for nabla_build_mask (same
 *               workspace size).
 * Errors: NABLA_ERR_INVALID_ARG as for nabla_build_mask, and for a negative
 * or non-finite topk_ratio.
 */
nabla_status nabla_build_mask_topk(const void *q, const void *k, nabla_dtype dt, int B, int S,
                                   int h, int D, double topk_ratio, int32_t *kv_nb,
                                   int32_t *kv_inds, void *workspace, size_t ws_bytes,
                                   nabla_stream_t stream);

/*
 * nabla_attn_fwd -- block-sparse attention forward over the kept 64x64 blocks
 * ([P1] NablaAttentionImpl.forward: flex_attention with a BlockMask of full
 * 64x64 blocks, non-causal; [P4] Expansion).
 *
 * For every (b, hh, query token s in block i), with J the tokens of the blocks
 * kv_inds[b, hh, i, 0 .. kv_nb[b, hh, i]-1]:
 *   o[b, s, hh, :] = sum_{u in J} softmax_u( scale * <q_s, k_u> ) v_u,
 * computed with an online softmax in fp32; o = 0 for a row with kv_nb = 0.
 * bf16: QK^T and PV run on the tcgen05 tensor cores (bf16 operands, fp32
 * accumulators; P is rounded to bf16 before PV); o is written as bf16.
 * f32: fp32 CUDA-core arithmetic throughout; o is written as fp32.
 * Results are reproducible bit for bit: on a given GPU model, repeated calls on
 * the same inputs give the same o (and lse).  The order in which a row's kept
 * blocks are accumulated depends only on kv_nb, kv_inds and the number of SMs,
 * never on timing.
 *
 *   q, k, v, o  [B, S, h, D] device, element type dt; o is overwritten.
 *   kv_nb       [B, h, s1] device int32, each in [0, s1].
 *   kv_inds     [B, h, s1, s1] device int32; the first kv_nb entries of each row
 *               are block indices in [0, s1), strictly ascending.
 *   scale       softmax scale (normally 1/sqrt(D), flex_attention's default).
 * Out-of-range kv_nb / kv_inds entries are skipped and reported as
 * NABLA_ERR_BAD_INDEX by nabla_get_last_device_status; they never cause an
 * out-of-bounds access.
 * Errors: NABLA_ERR_INVALID_ARG as for nabla_build_mask (shape, dtype,
 * pointers) and for a non-finite scale.
 */
nabla_status nabla_attn_fwd(const void *q, const void *k, const void *v, nabla_dtype dt, int B,
                            int S, int h, int D, const int32_t *kv_nb, const int32_t *kv_inds,
                            float scale, void *o, nabla_stream_t stream);

/*
 * nabla_attn_fwd_lse -- nabla_attn_fwd that also writes, for every query row,
 * the base-2 log-sum-exp of its scaled scores over the kept tokens J:
 *   lse[(b*h + hh)*S + s] = log2( sum_{u in J} 2^(scale * log2(e) * <q_s, k_u>) ),
 * or -INFINITY for a row whose block keeps nothing.  A training step stores it
 * for nabla_attn_bwd, which then needs no pass of its own to renormalise P.
 *   lse  [B, h, S] device fp32, 4-byte aligned, written (NULL is rejected).
 * Everything else, including o, is exactly as nabla_attn_fwd.
 */
nabla_status nabla_attn_fwd_lse(const void *q, const void *k, const void *v, nabla_dtype dt,
                                int B, int S, int h, int D, const int32_t *kv_nb,
                                const int32_t *kv_inds, float scale, void *o, float *lse,
                                nabla_stream_t stream);

/*
 * nabla_attn_bwd -- gradients of nabla_attn_fwd with respect to q, k and v
 * (gist.science NABLA summary, "Dual-Phase Acceleration" and Experimental
 * Results: the method trains with the block mask, so the forward is
 * differentiated; [P1] NablaAttentionImpl.forward is the function).
 *
 * For every (b, hh) and query token s in block i, J the tokens of the kept
 * blocks of row i, z_su = scale <q_s, k_u>, P = softmax_u(z), and the upstream
 * gradient dout:
 *   dv_u = sum_s P_su dout_s              dP_su = <dout_s, v_u>
 *   delta_s = <dout_s, o_s>               dz_su = P_su (dP_su - delta_s)
 *   dq_s = scale sum_u dz_su k_u          dk_u = scale sum_s dz_su q_s
 * where the sums over s run over every query row whose block kept u's block.
 * Rows with kv_nb = 0 contribute nothing (their dq is 0); key blocks that no
 * row kept get dk = dv = 0.  delta is formed from the o passed in, which
 * must be the forward output for the same inputs (as stored by a training
 * step).  fp32 storage: fp32 arithmetic on CUDA cores.  bf16 storage: the
 * products run on tcgen05 with fp32 accumulation; P and dz enter the products
 * as bf16, as the forward's P does.  dq, dk, dv are written in dt.
 *
 *   q, k, v, o, dout  [B, S, h, D] device, element type dt.
 *   lse               [B, h, S] device fp32 (16-byte aligned) from
 *                     nabla_attn_fwd_lse for the same inputs, or NULL: the
 *                     library then computes it (bf16: one tcgen05 forward;
 *                     fp32: a pass over the kept blocks on CUDA cores).
 *   kv_nb, kv_inds    the mask, as for nabla_attn_fwd (bad entries are skipped
 *                     and reported as NABLA_ERR_BAD_INDEX).
 *   scale             the forward's softmax scale.
 *   dq, dk, dv        [B, S, h, D] device, element type dt, overwritten.
 *   workspace         device scratch of ws_bytes >= nabla_attn_bwd_workspace_bytes()
 *                     (256-byte aligned): the rows' log-sum-exp and delta, the
 *                     transposed mask (for each key block, the query blocks
 *                     that kept it), and a bf16 o-sized scratch used when dt is
 *                     bf16 and lse is NULL (the library then runs the tcgen05
 *                     forward once to obtain lse).
 * Errors: NABLA_ERR_INVALID_ARG as for nabla_attn_fwd, for NULL or unaligned
 * o, dout, dq, dk, dv or workspace, an lse not 16-byte aligned, and a short
 * workspace.
 */
size_t nabla_attn_bwd_workspace_bytes(int B, int S, int h, int D);
nabla_status nabla_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dout, nabla_dtype dt, int B, int S,
                            int h, int D,
                            const int32_t *kv_nb, const int32_t *kv_inds, float scale, void *dq,
                            void *dk, void *dv, void *workspace, size_t ws_bytes,
                            nabla_stream_t stream);

/*
 * nabla_sta_mask -- the spatio-temporal window ([P1] NablaAttentionMetadata
 * "sta_mask"; [P4] Hybrid Integration with STA).  The pages do not show its
 * construction; this library's reading: on the (T, H, W) block grid with
 * block index (t*H + y)*W + x, sta[i*s1 + j] = 1 iff |t_i - t_j| <= wt,
 * |y_i - y_j| <= wh and |x_i - x_j| <= ww (no wrap-around), else 0.
 *   sta   [s1, s1] device uint8 with s1 = T*H*W <= 2048, written.
 * Errors: NABLA_ERR_INVALID_ARG for T, H, W < 1, s1 > 2048, negative half
 * widths, NULL sta.
 */
nabla_status nabla_sta_mask(int T, int H, int W, int wt, int wh, int ww, uint8_t *sta,
                            nabla_stream_t stream);

/*
 * nabla_fractal_flatten / nabla_fractal_unflatten -- the token order the path
 * expects ([P4] Methodology, "Token Reordering (Fractal Flattening)": the tokens
 * of each P x P spatial patch are grouped into a contiguous run, the temporal
 * order is kept; [P1] forward: q/k/v arrive "fractal-ordered by the model" and
 * nablaT_v2 pools 64-token blocks, so with P = 8 each block is one patch of
 * one frame).  This library's reading of the order: frames in time order, the
 * patches of a frame in raster order, the tokens of a patch row-major:
 *   fractal token ((t*(H/P) + py)*(W/P) + px)*P*P + yi*P + xi
 *   = raster token (t*H + py*P + yi)*W + px*P + xi.
 *
 *   x  [B, T, H, W, h, D] device, tokens in (t, y, x) raster order.
 *   y  [B, T*H*W, h, D] device, tokens in fractal order.
 * flatten reads x and writes y; unflatten reads y and writes x (the inverse,
 * for the attention output).  A token's h*D elements move as one row, so any
 * dtype works; dt fixes the element size (2 bytes bf16, 4 bytes f32).
 * The two buffers must not overlap.  Asynchronous on `stream`.
 * Errors: NABLA_ERR_INVALID_ARG for B, T, H, W, h, D or P < 1, H or W not a
 * multiple of P, h*D*element size not a multiple of 16 bytes, NULL, unaligned
 * (16 bytes) or overlapping buffers, an unknown dtype.
 */
nabla_status nabla_fractal_flatten(const void *x, nabla_dtype dt, int B, int T, int H, int W,
                                   int h, int D, int P, void *y, nabla_stream_t stream);
nabla_status nabla_fractal_unflatten(const void *y, nabla_dtype dt, int B, int T, int H, int W,
                                     int h, int D, int P, void *x, nabla_stream_t stream);

/*
 * Diagnostic of the failure-detection path (no counterpart on the pages):
 * enqueues one CTA that waits on an mbarrier nothing ever arrives on, through
 * the same bounded wait the attention kernel uses, with a 20 ms limit.  The
 * wait gives up and records NABLA_ERR_TIMEOUT in the device status word; the
 * context stays usable.  Returns NABLA_OK when the probe was launched.
 */
nabla_status nabla_selftest_bounded_wait(nabla_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status words that
 * the kernels above set (bounded-wait timeouts, skipped out-of-range indices).
 * Returns NABLA_OK when nothing was recorded, NABLA_ERR_CUDA when the
 * synchronisation itself failed, else the first recorded condition.
 */
nabla_status nabla_get_last_device_status(nabla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NABLA_H */
