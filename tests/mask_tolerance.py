"""Which differences between the float32 CUDA mask and the fp64 oracle mask are admissible.

Test infrastructure, like the oracle it reads.

The stated criterion: kv_nb and kv_inds are bit-exact except for blocks whose oracle
running sum lies within 1e-4 of 1 - thr (FastVideo API reference, page "nabla",
nablaT_v2 "Map binarization": keep when the ascending running sum is >= 1 - thr).
Those "window" blocks come from the oracle's `ambiguous_blocks`.

Reading R8(b) adds near ties that straddle the cut.  Two blocks a (CDF-dropped) and b
(CDF-kept) of a row whose probabilities are closer than the CUDA path can resolve may
come out in the other order; a swap moves each running sum by a whole block mass, so
both may differ from the oracle although neither is in the window.  How close "closer
than the CUDA path can resolve" is follows from that path's arithmetic, per block:

  The device orders blocks of a row by e_j = 2^(L~_j - M~), where L~_j is its float32
  base-2 logit (log2 e / sqrt(D)) <qa_i, ka_j> and M~ the row maximum.  M~ is common to
  the row, so the order of a and b flips only if
      |p_a - p_b| <= (theta_a + theta_b) max(p_a, p_b),
      theta_j = ln 2 (U_j + 2^-24 |L_j - M|) + EPS_EX2,
  with U_j a bound on |L~_j - L_j| and EPS_EX2 the relative error of the device's
  2^x.  `logit_error_bound` derives U from the kernels' arithmetic (its docstring lists
  each term); a GPU test checks the device's pooled map against it entry by entry.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import nabla_oracle as O

U24 = 2.0 ** -24  # unit roundoff of float32 (round to nearest)
U23 = 2.0 ** -23  # one float32 ulp at 1: the error of one truncating accumulation step
U22 = 2.0 ** -22  # the residual of a two-part tf32 split (2^-11 of 2^-11)
# 2^x on the device (ex2.approx): the PTX ISA documents a maximum relative error of
# about 2^-22 for the f32 form; twice that is taken.
EPS_EX2 = 2.0 ** -21
# Pooling: a block mean is a sum of 64 values in float32, then a scale.  The CUDA-core
# pool adds 16 rows per thread (15 rounded additions), joins four partial sums (3) and
# scales (1): at most 19 roundings, each below U24 * sum|x|, so 19 U24 of the block mean
# of |x|.  The tensor-core pool sums the 64 rows in four K=16 MMA steps into an fp32
# accumulator; a step that aligns and truncates each of its 16 products and the
# accumulator errs by at most 17 U23 of its magnitude sum, so 34 U24 of the mean of
# |x| in all, plus the scale.  C_POOL covers both pools.
C_POOL = 36 * U24
# Map: three tf32 MMA terms (lo_q hi_k, hi_q lo_k, hi_q hi_k) per 8-wide k-step.  The
# two-part split leaves U22 |m| of each mean (q and k), and the dropped lo_q lo_k term is
# below U22 |q k|: 3 U22 per product.  Each of the 3 D / 8 MMA k-steps adds into the
# fp32 accumulator with at most one truncation of U23 times the accumulator plus its
# products' magnitudes, which sum to at most (3 D / 8 + 1) U23 sum_d |q_d k_d|.
def c_map(D: int) -> float:
    return 3 * U22 + (3 * D // 8 + 1) * U23


def logit_error_bound(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """U[b, h, i, j] >= |L~_ij - L_ij|, in base-2 logit units, for q, k [B, S, h, D].

    Terms (s = log2(e) / sqrt(D), a = block mean of |x|):
      pooling:  the means carry C_POOL * a_d of error per component (q and k), which
                reaches the logit as s * sum_d (C_POOL a^q_d |ka_d| + |qa_d| C_POOL a^k_d);
      map:      s * c_map(D) * sum_d |qa_d| |ka_d| (split residuals, dropped lo*lo term,
                accumulation roundings);
      scaling:  the q means are scaled by s in float32 before the split (one more U24 of
                |qa_d| in every term, folded into the map coefficient).
    """
    D = q.shape[-1]
    s = math.log2(math.e) / math.sqrt(D)
    qa = np.abs(O.pool_blocks(q))
    ka = np.abs(O.pool_blocks(k))
    aq = O.pool_blocks(np.abs(q))
    ak = O.pool_blocks(np.abs(k))
    kt = np.swapaxes(ka, -1, -2)
    pool = C_POOL * (np.matmul(aq, kt) + np.matmul(qa, np.swapaxes(ak, -1, -2)))
    prod = (c_map(D) + U24) * np.matmul(qa, kt)
    return s * (pool + prod)


def block_margins(q: np.ndarray, k: np.ndarray, p: np.ndarray) -> np.ndarray:
    """theta[b, h, i, j]: the relative error bound of the device's e_j (see module doc).

    p: the oracle's softmax rows, from which |L_j - M| = -log2(p_j / max p) is taken."""
    U = logit_error_bound(q, k)
    with np.errstate(divide="ignore"):
        depth = -np.log2(p / p.max(axis=-1, keepdims=True))
    depth = np.where(np.isfinite(depth), depth, 0.0)
    return math.log(2.0) * (U + U24 * depth) + EPS_EX2


def near_tie_blocks(p: np.ndarray, cdf_mask: np.ndarray, theta, sta=None) -> np.ndarray:
    """Blocks in a near tie straddling the cut (reading R8(b)).

    A CDF-dropped block j is flagged when the lightest CDF-kept block k of its row is
    within (theta_j + theta_k) max(p_j, p_k) of it; a CDF-kept block when the heaviest
    CDF-dropped block is.  STA blocks are never flagged (they are kept whatever the
    order) but serve as partners.  theta: scalar or array broadcastable to p."""
    theta = np.broadcast_to(np.asarray(theta, dtype=np.float64), p.shape)
    dropped = ~cdf_mask
    inf = np.inf
    kmin = np.argmin(np.where(cdf_mask, p, inf), axis=-1)[..., None]
    dmax = np.argmax(np.where(dropped, p, -inf), axis=-1)[..., None]
    has_k = cdf_mask.any(axis=-1, keepdims=True)
    has_d = dropped.any(axis=-1, keepdims=True)
    pk = np.take_along_axis(p, kmin, -1)
    tk = np.take_along_axis(theta, kmin, -1)
    pd = np.take_along_axis(p, dmax, -1)
    td = np.take_along_axis(theta, dmax, -1)
    flag_d = dropped & has_k & (pk - p <= (theta + tk) * np.maximum(p, pk))
    flag_k = cdf_mask & has_d & (p - pd <= (theta + td) * np.maximum(p, pd))
    out = flag_d | flag_k
    if sta is not None:
        out &= ~np.asarray(sta, dtype=bool)  # [s1] or [s1, s1]: broadcasts over the rows
    return out


def mismatch_report(got: np.ndarray, ref: dict, window: np.ndarray, ties: np.ndarray,
                    theta: np.ndarray, limit: int = 40):
    """Per mismatched block: its oracle running sum relative to the cut, its probability,
    the relative gap to its partner across the cut and the pair's margin.  Returns the
    rows as dicts (first `limit`) and summary figures."""
    mism = got != ref["mask"]
    p, c, t, cdf = ref["p"], ref["c"], ref["t"], ref["cdf_mask"]
    rows = []
    worst_ratio = 0.0
    for idx in zip(*np.nonzero(mism)):
        row = idx[:-1]
        pr, cr, tr = p[row], cdf[row], theta[row]
        j = idx[-1]
        if cr[j]:
            cand = np.where(~cr, pr, -np.inf)
        else:
            cand = np.where(cr, pr, np.inf)
        k = int(np.argmin(np.abs(cand - pr[j])))
        gap = abs(pr[j] - pr[k]) / max(pr[j], pr[k]) if np.isfinite(cand[k]) else np.inf
        margin = tr[j] + tr[k]
        in_window = bool(window[idx])
        if not in_window and np.isfinite(gap):
            worst_ratio = max(worst_ratio, gap / margin)
        if len(rows) < limit:
            rows.append({"block": tuple(int(x) for x in idx), "c_minus_t": float(c[idx] - t),
                         "p": float(pr[j]), "partner": int(k), "rel_gap": float(gap),
                         "margin": float(margin), "window": in_window,
                         "near_tie": bool(ties[idx]), "oracle_kept": bool(ref["mask"][idx])})
    return rows, {"mismatches": int(mism.sum()),
                  "in_window": int((mism & window).sum()),
                  "near_tie_only": int((mism & ties & ~window).sum()),
                  "outside_window": int((mism & ~window).sum()),
                  "worst_gap_over_margin": float(worst_ratio)}
