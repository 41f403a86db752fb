"""NABLA oracle: a plain, slow, float64 CPU statement of what the hot path computes.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
CPU-baseline leg of the benchmark may import this module. The product path
(the CUDA library and its Python binding) never calls it and has no CPU
fallback.

Sources (the pages this restates):
  [P1] FastVideo API reference, page "nabla" (fastvideo.attention.backends.nabla):
       function nablaT_v2 -- "Map estimation" and "Map binarization" steps and the
       BlockMask creation; NablaAttentionImpl.forward -- flex_attention over the
       block mask on [B, S, heads, head_dim] inputs; NablaAttentionMetadata --
       the STA window mask is a block-level [1, 1, S/64, S/64] tensor.
  [P4] "NABLA: Neighborhood Adaptive Block-Level Attention" (gist.science
       technical summary), Methodology: Downsampling, Reduced Attention, CDF
       Thresholding, Expansion, Hybrid Integration with STA (M = M_nabla OR M_STA).

Readings taken where the pages are silent or differ (each also listed in the
design notes):
  R1 precision: everything here is float64; the pages' bf16 intermediates are
     not reproduced.
  R2 ties in the ascending sort are broken by lower block index first.
  R3 kept KV block indices are listed in ascending order; the tail of the
     index row after kv_nb entries is unspecified (filled with -1 here).
  R4 the comparison is "cumulative >= 1 - thr" ([P1] code), not [P4]'s "exceeds".
  R5 thr must lie in (0, 1].
  R6 a query block with no kept KV block produces a zero output row.
  R7 the STA window keeps block j for row i iff |dt| <= wt, |dy| <= wh and
     |dx| <= ww on the (T, H, W) block grid, raster order, no wrap-around.
  R14 top-k selector: ties in the score at the k-th place go to the higher
     block index (the kept set is the last k of the ascending (score, index)
     order, as in R2); topk = min(s1, floor(topk_ratio * s1)).
  R13 fractal flattening is one level of P x P patches: frames in time order,
     the patches of a frame in raster order, the tokens of a patch row-major;
     H and W must be multiples of P (with P = 8 each 64-token block is one
     patch of one frame).
  R17 backward: delta_s = dout_s . o_s is formed from the o passed in (the
     stored forward output) when one is given, else from the exact o.

Parity pins: every function below is pinned by tests that do not reuse its
own formula (closed forms, brute force, invariants, independent library
routines, and hand-worked fixtures in tests/golden/). No function here is
"parity unpinned".
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np

BLOCK = 64


# ---------------------------------------------------------------------------
# a1: block mean-pool.  [P1] nablaT_v2 "Map estimation": q and k are viewed as
# [B, h, S/64, 64, D] and averaged over the 64 tokens of each block.
# [P4] Methodology, "Downsampling".
# ---------------------------------------------------------------------------
def pool_blocks(x: np.ndarray) -> np.ndarray:
    """Mean of each 64-token block.

    x: real array [B, S, h, D] (any float dtype; widened to float64 block by block).
    returns float64 [B, h, S/64, D].
    """
    B, S, h, D = x.shape
    if S % BLOCK:
        raise ValueError("S must be a multiple of 64")
    s1 = S // BLOCK
    out = np.empty((B, h, s1, D), dtype=np.float64)
    step = max(1, (1 << 22) // max(1, BLOCK * h * D))  # blocks per chunk
    for i0 in range(0, s1, step):
        i1 = min(s1, i0 + step)
        chunk = x[:, i0 * BLOCK:i1 * BLOCK].astype(np.float64)
        chunk = chunk.reshape(B, i1 - i0, BLOCK, h, D)
        total = np.zeros((B, i1 - i0, h, D), dtype=np.float64)
        for r in range(BLOCK):
            total += chunk[:, :, r]
        out[:, :, i0:i1, :] = (total / BLOCK).transpose(0, 2, 1, 3)
    return out


# ---------------------------------------------------------------------------
# a2: pooled map.  [P1] nablaT_v2: map = qa @ ka^T, then divided by sqrt(D)
# (D = head dim) before the softmax.  [P4] "Reduced Attention".
# ---------------------------------------------------------------------------
def pooled_logits(qa: np.ndarray, ka: np.ndarray) -> np.ndarray:
    """L[b, h, i, j] = <qa[b,h,i], ka[b,h,j]> / sqrt(D), float64."""
    D = qa.shape[-1]
    return np.matmul(qa, np.swapaxes(ka, -1, -2)) / math.sqrt(D)


# ---------------------------------------------------------------------------
# a3: row softmax of the pooled map ([P1] nablaT_v2, softmax over the last dim).
# ---------------------------------------------------------------------------
def softmax_rows(L: np.ndarray) -> np.ndarray:
    m = L.max(axis=-1, keepdims=True)
    e = np.exp(L - m)
    return e / e.sum(axis=-1, keepdims=True)


# ---------------------------------------------------------------------------
# a4: CDF binarisation.  [P1] nablaT_v2 "Map binarization": sort each row
# ascending, take the running sum, keep entries whose running sum is >= 1-thr,
# and put the flags back in block order.  [P4] "CDF Thresholding".
# ---------------------------------------------------------------------------
def cdf_values(p: np.ndarray) -> np.ndarray:
    """c[..., j] = running sum of the row in ascending (p, j) order, up to and
    including block j (reading R2: ties by lower index first).  float64."""
    order = np.argsort(p, axis=-1, kind="stable")  # stable: equal p keep index order
    sorted_p = np.take_along_axis(p, order, axis=-1)
    run = np.cumsum(sorted_p, axis=-1)  # sequential accumulation along the row
    c = np.empty_like(run)
    np.put_along_axis(c, order, run, axis=-1)
    return c


def cut_level(thr: float) -> float:
    """t = 1 - thr in float64 (reading R5: thr in (0, 1])."""
    if not (0.0 < thr <= 1.0):
        raise ValueError("thr must lie in (0, 1]")
    return 1.0 - thr


def cdf_keep(p: np.ndarray, thr: float) -> np.ndarray:
    """Boolean CDF part of the mask: c(j) >= 1 - thr (reading R4)."""
    return cdf_values(p) >= cut_level(thr)


# ---------------------------------------------------------------------------
# a5: STA window.  [P1] NablaAttentionMetadata: block-level window mask shared
# by every batch and head; its construction is not shown (reading R7).
# [P4] "Hybrid Integration with STA".
# ---------------------------------------------------------------------------
def sta_mask(T: int, H: int, W: int, wt: int, wh: int, ww: int) -> np.ndarray:
    """uint8 [s1, s1] with s1 = T*H*W; block index (t*H + y)*W + x."""
    t, y, x = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    t, y, x = t.ravel(), y.ravel(), x.ravel()
    keep = ((np.abs(t[:, None] - t[None, :]) <= wt)
            & (np.abs(y[:, None] - y[None, :]) <= wh)
            & (np.abs(x[:, None] - x[None, :]) <= ww))
    return keep.astype(np.uint8)


# ---------------------------------------------------------------------------
# a6: union and CSR.  [P1] nablaT_v2: logical OR with the STA mask, kv_nb is
# the row count, kv_inds lists the kept blocks first (reading R3: ascending).
# ---------------------------------------------------------------------------
def csr_from_mask(mask: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """mask bool [..., s1, s1] -> (kv_nb int32 [..., s1], kv_inds int32 [..., s1, s1]).
    kv_inds rows hold the kept indices ascending, then -1."""
    mask = np.asarray(mask, dtype=bool)
    s1 = mask.shape[-1]
    kv_nb = mask.sum(axis=-1).astype(np.int32)
    cols = np.broadcast_to(np.arange(s1, dtype=np.int64), mask.shape)
    # kept columns keep their index as key, dropped ones go past the end
    key = np.where(mask, cols, s1 + cols)
    srt = np.sort(key, axis=-1)
    kv_inds = np.where(srt < s1, srt, -1).astype(np.int32)
    return kv_nb, kv_inds


def build_mask(q: np.ndarray, k: np.ndarray, sta: np.ndarray, thr: float):
    """The whole mask builder (a1..a6).

    q, k: [B, S, h, D] real arrays; sta: [s1, s1] 0/1; thr in (0, 1].
    returns dict: kv_nb, kv_inds, mask (bool [B,h,s1,s1]), cdf_mask, c (float64
    running sums), t (float64 cut level), p (softmax rows).
    """
    qa = pool_blocks(q)
    ka = pool_blocks(k)
    p = softmax_rows(pooled_logits(qa, ka))
    c = cdf_values(p)
    t = cut_level(thr)
    cdf_mask = c >= t
    mask = np.logical_or(cdf_mask, np.asarray(sta, dtype=bool)[None, None])
    kv_nb, kv_inds = csr_from_mask(mask)
    return {"kv_nb": kv_nb, "kv_inds": kv_inds, "mask": mask, "cdf_mask": cdf_mask,
            "c": c, "t": t, "p": p}


def ambiguous_blocks(c: np.ndarray, t: float, sta: Optional[np.ndarray] = None,
                     tol: float = 1e-4) -> np.ndarray:
    """Blocks whose running sum lies within tol of the cut level and that the STA
    does not force on: the window of the stated mask tolerance, where a float32
    device result may differ.  sta ([s1] for one row, [s1, s1] for a map) broadcasts
    over the leading axes of c."""
    amb = np.abs(c - t) < tol
    if sta is not None:
        amb &= ~np.asarray(sta, dtype=bool)
    return amb


# ---------------------------------------------------------------------------
# a7: block-sparse attention.  [P1] NablaAttentionImpl.forward: flex_attention
# with the block mask (64x64 blocks, all full blocks, default scale, non-causal).
# [P4] "Expansion": the block mask selects which 64x64 blocks are computed.
# The plain definition is masked dense softmax attention restricted to the
# kept blocks; reading R6 for rows with nothing kept.
# ---------------------------------------------------------------------------
def block_sparse_attention(q, k, v, kv_nb, kv_inds, scale: float,
                           qblocks: Optional[Iterable[Tuple[int, int, int]]] = None):
    """o[b, s, h, :] for the query blocks listed in qblocks (all if None).

    q, k, v: real [B, S, h, D]; kv_nb [B, h, s1]; kv_inds [B, h, s1, s1].
    returns float64 [B, S, h, D] (rows of unlisted blocks are NaN) when qblocks
    is None or given; always a full-shape array.
    """
    B, S, h, D = q.shape
    s1 = S // BLOCK
    out = np.full((B, S, h, D), np.nan, dtype=np.float64)
    if qblocks is None:
        qblocks = [(b, hh, i) for b in range(B) for hh in range(h) for i in range(s1)]
    for b, hh, i in qblocks:
        n = int(kv_nb[b, hh, i])
        rows = slice(i * BLOCK, (i + 1) * BLOCK)
        if n == 0:
            out[b, rows, hh, :] = 0.0
            continue
        blocks = np.asarray(kv_inds[b, hh, i, :n], dtype=np.int64)
        # the kept blocks' tokens, block by block in list order (64 rows each)
        Q = q[b, rows, hh, :].astype(np.float64)
        K = np.asarray(k[b, :, hh, :].reshape(s1, BLOCK, D)[blocks].reshape(-1, D), np.float64)
        V = np.asarray(v[b, :, hh, :].reshape(s1, BLOCK, D)[blocks].reshape(-1, D), np.float64)
        a = scale * (Q @ K.T)
        a -= a.max(axis=1, keepdims=True)
        e = np.exp(a)
        out[b, rows, hh, :] = (e @ V) / e.sum(axis=1, keepdims=True)
    return out


def attention_lse2(q, k, kv_nb, kv_inds, scale: float,
                   qblocks: Optional[Iterable[Tuple[int, int, int]]] = None):
    """Base-2 log-sum-exp of each query row's scaled scores over its kept tokens,
    log2(sum_u 2^(scale log2(e) <q_s, k_u>)) = (natural log-sum-exp) / ln 2;
    float64 [B, h, S], -inf for rows whose block keeps nothing, NaN for rows of
    unlisted blocks."""
    B, S, h, D = q.shape
    s1 = S // BLOCK
    out = np.full((B, h, S), np.nan, dtype=np.float64)
    if qblocks is None:
        qblocks = [(b, hh, i) for b in range(B) for hh in range(h) for i in range(s1)]
    for b, hh, i in qblocks:
        n = int(kv_nb[b, hh, i])
        rows = slice(i * BLOCK, (i + 1) * BLOCK)
        if n == 0:
            out[b, hh, rows] = -np.inf
            continue
        blocks = np.asarray(kv_inds[b, hh, i, :n], dtype=np.int64)
        tok = (blocks[:, None] * BLOCK + np.arange(BLOCK)[None, :]).ravel()
        z = scale * (q[b, rows, hh, :].astype(np.float64) @ k[b, tok, hh, :].astype(np.float64).T)
        m = z.max(axis=1)
        out[b, hh, rows] = (m + np.log(np.exp(z - m[:, None]).sum(axis=1))) / math.log(2.0)
    return out


# ---------------------------------------------------------------------------
# Backward of a7 (training).  gist.science NABLA summary, "Dual-Phase
# Acceleration" and Experimental Results (pre-training iteration time): the
# method is used for training, where flex_attention ([P1] forward) is
# differentiated by autograd.  The plain definition is the gradient of the
# masked softmax attention of a7 with respect to q, k and v, for an upstream
# gradient dout of o.  With z = scale * q k^T over the kept tokens J of a row,
# P = softmax(z), o = P v:
#   dv_u = sum_s P_su dout_s            dP_su = dout_s . v_u
#   delta_s = sum_u P_su dP_su = dout_s . o_s
#   dz_su = P_su (dP_su - delta_s)
#   dq_s = scale sum_u dz_su k_u        dk_u = scale sum_s dz_su q_s
# Rows with nothing kept (R6) contribute nothing.  Reading R17: when o is
# passed, delta_s is formed from that o (dout_s . o_s), as a training step
# does with the forward output it stored; otherwise from the exact o.
# ---------------------------------------------------------------------------
def block_sparse_attention_bwd(q, k, v, dout, kv_nb, kv_inds, scale: float, o=None,
                               qblocks: Optional[Iterable[Tuple[int, int, int]]] = None):
    """(dq, dk, dv), float64 [B, S, h, D] each.

    qblocks restricts the sums over query rows to the listed (b, h, i) blocks:
    dq is then exact for those blocks (0 elsewhere), and dk, dv of a key block
    are exact when every block that kept it is listed."""
    B, S, h, D = q.shape
    s1 = S // BLOCK
    dq = np.zeros((B, S, h, D), dtype=np.float64)
    dk = np.zeros((B, S, h, D), dtype=np.float64)
    dv = np.zeros((B, S, h, D), dtype=np.float64)
    if qblocks is None:
        qblocks = [(b, hh, i) for b in range(B) for hh in range(h) for i in range(s1)]
    for b, hh, i in qblocks:
        n = int(kv_nb[b, hh, i])
        if n == 0:
            continue
        rows = slice(i * BLOCK, (i + 1) * BLOCK)
        blocks = np.asarray(kv_inds[b, hh, i, :n], dtype=np.int64)
        tok = (blocks[:, None] * BLOCK + np.arange(BLOCK)[None, :]).ravel()
        Q = q[b, rows, hh, :].astype(np.float64)
        K = k[b, tok, hh, :].astype(np.float64)
        V = v[b, tok, hh, :].astype(np.float64)
        dO = dout[b, rows, hh, :].astype(np.float64)
        z = scale * (Q @ K.T)
        z -= z.max(axis=1, keepdims=True)
        P = np.exp(z)
        P /= P.sum(axis=1, keepdims=True)
        O = P @ V if o is None else o[b, rows, hh, :].astype(np.float64)
        dP = dO @ V.T
        delta = (dO * O).sum(axis=1, keepdims=True)
        dz = P * (dP - delta)
        dq[b, rows, hh, :] = scale * (dz @ K)
        dk[b, tok, hh, :] += scale * (dz.T @ Q)
        dv[b, tok, hh, :] += P.T @ dO
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Fractal flattening (the step before the path).  [P1] module description and
# NablaAttentionImpl.forward: q/k/v arrive "fractal-ordered by the model" and
# nablaT_v2 pools 64-token blocks of that order; [P4] Methodology, "Token
# Reordering (Fractal Flattening)": the tokens of each P x P spatial patch are
# made contiguous while the temporal order is kept.  Reading R13.
# ---------------------------------------------------------------------------
def fractal_flatten(x: np.ndarray, P: int) -> np.ndarray:
    """x [B, T, H, W, h, D] (tokens in (t, y, x) raster order) -> [B, T*H*W, h, D]
    in fractal order."""
    B, T, H, W = x.shape[:4]
    if H % P or W % P:
        raise ValueError("H and W must be multiples of P")
    y = x.reshape(B, T, H // P, P, W // P, P, *x.shape[4:])
    # (b, t, patch row, patch col, row in patch, col in patch, ...)
    y = np.transpose(y, (0, 1, 2, 4, 3, 5) + tuple(range(6, y.ndim)))
    return np.ascontiguousarray(y).reshape(B, T * H * W, *x.shape[4:])


def fractal_unflatten(y: np.ndarray, T: int, H: int, W: int, P: int) -> np.ndarray:
    """Inverse of fractal_flatten: [B, T*H*W, h, D] -> [B, T, H, W, h, D]."""
    B = y.shape[0]
    if H % P or W % P or y.shape[1] != T * H * W:
        raise ValueError("shape mismatch")
    x = y.reshape(B, T, H // P, W // P, P, P, *y.shape[2:])
    x = np.transpose(x, (0, 1, 2, 4, 3, 5) + tuple(range(6, x.ndim)))
    return np.ascontiguousarray(x).reshape(B, T, H, W, *y.shape[2:])


# ---------------------------------------------------------------------------
# Top-k block selector (a second selector over the pooled map).  FastVideo
# API reference, attention backends index, sla.get_block_map: the keys are
# smoothed (k minus its mean over the sequence, per batch, head and channel),
# q and the smoothed k are mean-pooled over 64-token blocks, the block score is
# their plain product (no scale, no softmax), and each query block keeps the
# topk = min(K, int(topk_ratio * K)) key blocks of largest score.  Reading R14
# for ties; the kept blocks are listed ascending (as R3).
# ---------------------------------------------------------------------------
def topk_scores(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """q, k [B, S, h, D] -> block scores [B, h, s1, s1] (fp64)."""
    kf = np.asarray(k, dtype=np.float64)
    arg_k = kf - kf.mean(axis=1, keepdims=True)  # smooth-k: mean over the sequence
    return np.matmul(pool_blocks(q), np.swapaxes(pool_blocks(arg_k), -1, -2))


def topk_count(s1: int, topk_ratio: float) -> int:
    return min(s1, int(topk_ratio * s1))


def topk_mask(q: np.ndarray, k: np.ndarray, topk_ratio: float):
    """Returns dict: kv_nb, kv_inds (ascending, -1 tail), mask, scores, topk."""
    sc = topk_scores(q, k)
    s1 = sc.shape[-1]
    kk = topk_count(s1, topk_ratio)
    order = np.argsort(sc, axis=-1, kind="stable")  # ascending (score, index)
    keep = np.zeros(sc.shape, dtype=bool)
    if kk > 0:
        np.put_along_axis(keep, order[..., s1 - kk:], True, axis=-1)
    kv_nb, kv_inds = csr_from_mask(keep)
    return {"kv_nb": kv_nb, "kv_inds": kv_inds, "mask": keep, "scores": sc, "topk": kk}

