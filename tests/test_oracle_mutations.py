"""Plant plausible mistakes in copies of the oracle's steps (CPU only) and check
that the pins catch every one of them.  A pin set that let one of these pass
would not be pinning the oracle to the pages."""
import math

import numpy as np
import pytest

import oracle_pins as P
from oracle import nabla_oracle as O


def _cdf_strict(p, thr):  # "exceeds" instead of ">="
    return O.cdf_values(p) > (1.0 - thr)


def _cdf_descending(p, thr):  # running sum over a descending sort
    return _desc_values(p) >= (1.0 - thr)


def _desc_values(p):
    order = np.argsort(-p, axis=-1, kind="stable")
    run = np.cumsum(np.take_along_axis(p, order, -1), -1)
    c = np.empty_like(run)
    np.put_along_axis(c, order, run, -1)
    return c


def _cdf_ties_high_first(p, thr):  # ties broken by higher index first
    rev = p[..., ::-1]
    c = O.cdf_values(rev)[..., ::-1]
    return c >= (1.0 - thr)


def _cdf_exclusive(p, thr):  # running sum excluding the block itself
    return (O.cdf_values(p) - p) >= (1.0 - thr)


def _cdf_uses_thr(p, thr):  # compares against thr instead of 1 - thr
    return O.cdf_values(p) >= thr


def _map_transposed(qa, ka):
    return np.matmul(ka, np.swapaxes(qa, -1, -2)) / math.sqrt(qa.shape[-1])


def _map_no_scale(qa, ka):
    return np.matmul(qa, np.swapaxes(ka, -1, -2))


def _map_scale_d(qa, ka):
    return np.matmul(qa, np.swapaxes(ka, -1, -2)) / qa.shape[-1]


def _softmax_cols(L):
    e = np.exp(L - L.max(axis=-2, keepdims=True))
    return e / e.sum(axis=-2, keepdims=True)


def _pool_wrong_layout(x):  # treats [B,S,h,D] as if it were [B,h,S,D]
    B, S, h, D = x.shape
    y = np.ascontiguousarray(x).reshape(B, h, S, D)
    return y.reshape(B, h, S // 64, 64, D).mean(3)


def _pool_sum(x):  # sum instead of mean
    return O.pool_blocks(x) * 64


def _pool_off_by_one(x):  # blocks start one token late
    return O.pool_blocks(np.roll(x, -1, axis=1))


def _sta_axes_swapped(T, H, W, wt, wh, ww):
    return O.sta_mask(T, H, W, ww, wh, wt)


def _sta_wrap(T, H, W, wt, wh, ww):
    t, y, x = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    t, y, x = t.ravel(), y.ravel(), x.ravel()
    dt = np.abs(t[:, None] - t[None, :])
    dt = np.minimum(dt, T - dt)
    keep = (dt <= wt) & (np.abs(y[:, None] - y[None, :]) <= wh) & (np.abs(x[:, None] - x[None, :]) <= ww)
    return keep.astype(np.uint8)


def _csr_descending(mask):
    nb, inds = O.csr_from_mask(mask)
    out = inds.copy()
    for idx in np.ndindex(nb.shape):
        n = nb[idx]
        out[idx][:n] = inds[idx][:n][::-1]
    return nb, out


def _attn_no_scale(q, k, v, nb, inds, scale, qblocks=None):
    return O.block_sparse_attention(q, k, v, nb, inds, 1.0, qblocks)


def _attn_skip_first_block(q, k, v, nb, inds, scale, qblocks=None):
    inds2 = inds.copy()
    nb2 = nb.copy()
    for idx in np.ndindex(nb.shape):
        if nb[idx] > 1:
            inds2[idx][: nb[idx] - 1] = inds[idx][1:nb[idx]]
            nb2[idx] -= 1
    return O.block_sparse_attention(q, k, v, nb2, inds2, scale, qblocks)


def _attn_empty_nan(q, k, v, nb, inds, scale, qblocks=None):
    o = O.block_sparse_attention(q, k, v, nb, inds, scale, qblocks)
    B, S, h, D = q.shape
    for b, hh, i in zip(*np.nonzero(nb == 0)):
        o[b, 64 * i:64 * (i + 1), hh] = np.nan
    return o


CDF_MUTANTS = [_cdf_strict, _cdf_descending, _cdf_ties_high_first, _cdf_exclusive, _cdf_uses_thr]


@pytest.mark.parametrize("mutant", CDF_MUTANTS, ids=lambda f: f.__name__)
def test_cdf_mutants_caught(mutant):
    caught = 0
    for check in (P.check_cdf_golden, P.check_cdf_bruteforce, P.check_cdf_invariants):
        try:
            check(mutant)
        except AssertionError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("mutant", [_map_transposed, _map_no_scale, _map_scale_d],
                         ids=lambda f: f.__name__)
def test_map_mutants_caught(mutant):
    with pytest.raises(AssertionError):
        P.check_map(mutant)


def test_softmax_mutant_caught():
    with pytest.raises(AssertionError):
        P.check_softmax(_softmax_cols)


@pytest.mark.parametrize("mutant", [_pool_wrong_layout, _pool_sum, _pool_off_by_one],
                         ids=lambda f: f.__name__)
def test_pool_mutants_caught(mutant):
    with pytest.raises(AssertionError):
        P.check_pool(mutant)


@pytest.mark.parametrize("mutant", [_sta_axes_swapped, _sta_wrap], ids=lambda f: f.__name__)
def test_sta_mutants_caught(mutant):
    with pytest.raises(AssertionError):
        P.check_sta_golden(mutant)


def test_csr_mutant_caught():
    with pytest.raises(AssertionError):
        P.check_csr(_csr_descending)


@pytest.mark.parametrize("mutant", [_attn_no_scale, _attn_skip_first_block, _attn_empty_nan],
                         ids=lambda f: f.__name__)
def test_attention_mutants_caught(mutant):
    caught = 0
    for check in (P.check_attention_dense, P.check_attention_masked,
                  P.check_attention_closed_form):
        try:
            check(mutant, O.csr_from_mask)
        except AssertionError:
            caught += 1
    assert caught > 0


# ---- fractal flattening: plausible mistakes and the pins that catch them
def _fractal_col_major(x, Pp):  # tokens of a patch column-major
    B, T, H, W = x.shape[:4]
    y = x.reshape(B, T, H // Pp, Pp, W // Pp, Pp, *x.shape[4:])
    y = np.transpose(y, (0, 1, 2, 4, 5, 3) + tuple(range(6, y.ndim)))
    return np.ascontiguousarray(y).reshape(B, T * H * W, *x.shape[4:])


def _fractal_patches_col_major(x, Pp):  # patches of a frame column-major
    B, T, H, W = x.shape[:4]
    y = x.reshape(B, T, H // Pp, Pp, W // Pp, Pp, *x.shape[4:])
    y = np.transpose(y, (0, 1, 4, 2, 3, 5) + tuple(range(6, y.ndim)))
    return np.ascontiguousarray(y).reshape(B, T * H * W, *x.shape[4:])


def _fractal_time_inside_patch(x, Pp):  # time interleaved into the patch runs
    B, T, H, W = x.shape[:4]
    y = x.reshape(B, T, H // Pp, Pp, W // Pp, Pp, *x.shape[4:])
    y = np.transpose(y, (0, 2, 4, 1, 3, 5) + tuple(range(6, y.ndim)))
    return np.ascontiguousarray(y).reshape(B, T * H * W, *x.shape[4:])


FRACTAL_MUTANTS = [_fractal_col_major, _fractal_patches_col_major, _fractal_time_inside_patch]


@pytest.mark.parametrize("mutant", FRACTAL_MUTANTS, ids=lambda f: f.__name__)
def test_fractal_mutants_caught(mutant):
    import test_oracle_fractal as TF

    caught = False
    for shape, order in TF._cases():
        T, H, W, Pp = shape
        x = np.arange(T * H * W).reshape(1, T, H, W, 1, 1)
        if mutant(x, Pp).ravel().tolist() != order:
            caught = True
    assert caught


# ---- top-k selector: plausible mistakes
def _topk_lower_index_kept(q, k, ratio):  # ties broken toward the lower index
    sc = O.topk_scores(q, k)
    s1 = sc.shape[-1]
    kk = O.topk_count(s1, ratio)
    order = np.argsort(-sc, axis=-1, kind="stable")  # descending, lower index first
    keep = np.zeros(sc.shape, bool)
    if kk:
        np.put_along_axis(keep, order[..., :kk], True, axis=-1)
    return keep


def _topk_rounded_count(q, k, ratio):  # round instead of int
    sc = O.topk_scores(q, k)
    s1 = sc.shape[-1]
    kk = min(s1, int(round(ratio * s1)))
    order = np.argsort(sc, axis=-1, kind="stable")
    keep = np.zeros(sc.shape, bool)
    if kk:
        np.put_along_axis(keep, order[..., s1 - kk:], True, axis=-1)
    return keep


def _topk_smallest(q, k, ratio):  # the k smallest scores
    sc = O.topk_scores(q, k)
    kk = O.topk_count(sc.shape[-1], ratio)
    order = np.argsort(sc, axis=-1, kind="stable")
    keep = np.zeros(sc.shape, bool)
    if kk:
        np.put_along_axis(keep, order[..., :kk], True, axis=-1)
    return keep


@pytest.mark.parametrize("mutant", [_topk_lower_index_kept, _topk_rounded_count, _topk_smallest],
                         ids=lambda f: f.__name__)
def test_topk_mutants_caught(mutant):
    qm = np.zeros((1, 1, 4, 2)); qm[..., 0] = 1.0
    km = np.zeros((1, 1, 4, 2)); km[..., 0] = [3, 1, 4, 1]
    rep = lambda m: np.repeat(np.transpose(m, (0, 2, 1, 3))[:, :, None], 64, axis=2).reshape(1, 256, 1, 2)
    q, k = rep(qm), rep(km)
    caught = any(not np.array_equal(mutant(q, k, r), O.topk_mask(q, k, r)["mask"])
                 for r in (0.5, 0.7, 0.75))
    assert caught


# ---- attention backward: plausible mistakes, each caught by the finite-difference pin
def _bwd_variant(kind, q, k, v, dout, nb, inds, scale):
    B, S, h, D = q.shape
    dq, dk, dv = (np.zeros((B, S, h, D)) for _ in range(3))
    for b in range(B):
        for hh in range(h):
            for i in range(S // 64):
                n = int(nb[b, hh, i])
                if n == 0:
                    continue
                rows = slice(64 * i, 64 * i + 64)
                tok = (inds[b, hh, i, :n][:, None] * 64 + np.arange(64)[None, :]).ravel()
                Q, K, V, dO = q[b, rows, hh], k[b, tok, hh], v[b, tok, hh], dout[b, rows, hh]
                z = scale * Q @ K.T
                P = np.exp(z - z.max(1, keepdims=True))
                P /= P.sum(1, keepdims=True)
                dP = dO @ V.T
                delta = (dP.sum(1, keepdims=True) if kind == "delta_from_dp"
                         else (dO * (P @ V)).sum(1, keepdims=True))
                dz = P * (delta - dP) if kind == "sign" else P * (dP - delta)
                dq[b, rows, hh] = scale * dz @ (V if kind == "dq_uses_v" else K)
                dk[b, tok, hh] += (1.0 if kind == "no_scale_dk" else scale) * dz.T @ Q
                dv[b, tok, hh] += P.T @ dO
    return dq, dk, dv


@pytest.mark.parametrize("kind", ["no_scale_dk", "delta_from_dp", "sign", "dq_uses_v"])
def test_backward_mutants_caught(kind):
    rng = np.random.default_rng(5)
    B, h, D, S = 1, 1, 4, 128
    q, k, v, dout = (rng.standard_normal((B, S, h, D)) for _ in range(4))
    nb = np.array([[[2, 1]]], np.int32)
    inds = np.array([[[[0, 1], [1, -1]]]], np.int32)
    scale = 0.6
    got = _bwd_variant(kind, q, k, v, dout, nb, inds, scale)
    eps = 1e-6

    def loss(qq, kk, vv):
        return float((dout * O.block_sparse_attention(qq, kk, vv, nb, inds, scale)).sum())

    caught = False
    for t, g in enumerate(got):
        for _ in range(12):
            ix = tuple(int(rng.integers(n)) for n in q.shape)
            args = [q.copy(), k.copy(), v.copy()]
            args[t][ix] += eps
            fp = loss(*args)
            args[t][ix] -= 2 * eps
            fm = loss(*args)
            if abs((fp - fm) / (2 * eps) - g[ix]) > 1e-5:
                caught = True
    assert caught
