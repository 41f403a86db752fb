"""Checks that pin the fp64 oracle to facts fixed by the NABLA pages and by
mathematics, not to its own formulas.

Each check takes the functions it examines as arguments, so the mutation
tests can hand it a deliberately broken variant and confirm that the check
fails.  Sources are cited per check:
  [P1] FastVideo API reference, page "nabla": nablaT_v2 (Map estimation,
       Map binarization, BlockMask creation), NablaAttentionImpl.forward,
       NablaAttentionMetadata.
  [P4] gist.science technical summary of "NABLA: Neighborhood Adaptive
       Block-Level Attention", Methodology.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ fixtures
def load_cdf_rows():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "cdf_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            if key == "p":
                cur = {"p": np.array([float(x) for x in val.split()])}
            elif key == "thr":
                cur["thr"] = float(val)
            elif key == "keep":
                cur["keep"] = np.array([int(x) for x in val.split()], dtype=bool)
                cases.append(cur)
    return cases


def load_sta_windows():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "sta_windows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line == "end":
                cur["mask"] = np.array(cur["rows"], dtype=np.uint8)
                cases.append(cur)
                cur = None
                continue
            key, val = line.split(":", 1)
            nums = [int(x) for x in val.split()]
            if key == "grid":
                cur = {"grid": tuple(nums), "rows": []}
            elif key == "half":
                cur["half"] = tuple(nums)
            elif key == "row":
                cur["rows"].append(nums)
    return cases


# ------------------------------------------------------------------ a1 pool
def check_pool(pool_blocks):
    """[P1] Map estimation: 64-token block means of [B, S, h, D] -> [B, h, S/64, D].
    Constructed input: token r of block i, head hh, dim d holds
    f(i, hh, d) + (r - 31.5); the offsets cancel, so the mean is f exactly."""
    B, h, D, s1 = 2, 3, 8, 5
    i = np.arange(s1)[:, None, None]
    hh = np.arange(h)[None, :, None]
    d = np.arange(D)[None, None, :]
    f = 1000.0 * i + 10.0 * hh + 0.25 * d  # [s1, h, D], all exact in binary
    r = np.arange(64) - 31.5
    x = f[None, :, None, :, :] + r[None, None, :, None, None]  # [1, s1, 64, h, D]
    x = np.broadcast_to(x, (B, s1, 64, h, D)).reshape(B, s1 * 64, h, D).copy()
    x[1] *= -2.0
    got = pool_blocks(x)
    want = np.stack([f.transpose(1, 0, 2), -2.0 * f.transpose(1, 0, 2)])
    assert got.shape == (B, h, s1, D)
    assert np.array_equal(got, want)
    # constant blocks give the constant
    c = np.full((1, 128, 2, 4), 0.3)
    assert np.allclose(pool_blocks(c), 0.3, rtol=0, atol=1e-15)


def check_pool_vs_torch(pool_blocks, seed=1):
    """Library cross-check: torch fp64 view [B,h,S/64,64,D] and mean over tokens."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((2, 320, 3, 16))
    t = torch.from_numpy(x).transpose(1, 2).reshape(2, 3, 5, 64, 16).mean(dim=3)
    assert np.allclose(pool_blocks(x), t.numpy(), rtol=0, atol=1e-14)


# ------------------------------------------------------------------ a2/a3 map + softmax
def check_map(pooled_logits):
    """[P1] map = qa @ ka^T, divided by sqrt(D) before the softmax.
    Constructed: qa_i = i * e0, ka_j = (j + 1) * e0 + 5 * e1 -> L_ij = i (j+1) / sqrt(D);
    asymmetric, so a transposed product fails; D = 16 makes sqrt(D) = 4 exact."""
    D, n = 16, 6
    qa = np.zeros((1, 1, n, D))
    ka = np.zeros((1, 1, n, D))
    qa[0, 0, :, 0] = np.arange(n)
    ka[0, 0, :, 0] = np.arange(n) + 1.0
    ka[0, 0, :, 1] = 5.0
    want = np.outer(np.arange(n), np.arange(n) + 1.0) / 4.0
    got = pooled_logits(qa, ka)
    assert np.array_equal(got[0, 0], want)


def check_softmax(softmax_rows):
    """Closed forms: logits (0, ln 3) -> (1/4, 3/4); rows sum to one; adding a constant
    to a row changes nothing; a large logit gap gives a one-hot row."""
    p = softmax_rows(np.array([[0.0, math.log(3.0)]]))
    assert np.allclose(p, [[0.25, 0.75]], rtol=0, atol=1e-15)
    rng = np.random.default_rng(2)
    L = rng.standard_normal((4, 33)) * 3
    p = softmax_rows(L)
    assert np.allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.allclose(softmax_rows(L + 7.5), p, rtol=0, atol=1e-14)
    q = softmax_rows(np.array([[0.0, 800.0, 0.0]]))
    assert np.allclose(q, [[0.0, 1.0, 0.0]], atol=1e-300)
    # ratio of two entries is exp of their logit gap
    assert np.allclose(p[:, 3] / p[:, 5], np.exp(L[:, 3] - L[:, 5]), rtol=1e-12)


def check_map_softmax_vs_torch(pooled_logits, softmax_rows, seed=3):
    """Library cross-check of map + softmax with torch fp64."""
    rng = np.random.default_rng(seed)
    qa = rng.standard_normal((2, 3, 7, 32))
    ka = rng.standard_normal((2, 3, 7, 32))
    want = torch.softmax(torch.from_numpy(qa) @ torch.from_numpy(ka).transpose(-1, -2)
                         / math.sqrt(32), dim=-1).numpy()
    assert np.allclose(softmax_rows(pooled_logits(qa, ka)), want, rtol=0, atol=1e-14)


# ------------------------------------------------------------------ a4 CDF cut
def check_cdf_golden(cdf_keep):
    for case in load_cdf_rows():
        got = cdf_keep(case["p"][None, :], case["thr"])[0]
        assert np.array_equal(got, case["keep"]), (case, got)


def check_cdf_bruteforce(cdf_keep, n=10, rows=40, seed=4):
    """Brute force on tiny rows: the kept set must be the heaviest subset among the
    smallest subsets whose mass exceeds thr (exact characterisation of keeping the
    ascending running sums >= 1 - thr; continuous random p, so no ties)."""
    rng = np.random.default_rng(seed)
    subsets = np.array(list(itertools.product([0, 1], repeat=n)), dtype=bool)  # [2^n, n]
    sizes = subsets.sum(1)
    for r in range(rows):
        alpha = [0.3, 1.0, 3.0][r % 3]
        p = rng.dirichlet(np.full(n, alpha))
        thr = [0.5, 0.7, 0.9, 0.95, 0.99][r % 5]
        mass = subsets.astype(np.float64) @ p
        ok = mass > thr
        mstar = sizes[ok].min()
        cand = np.where(ok & (sizes == mstar))[0]
        best = cand[np.argmax(mass[cand])]
        got = cdf_keep(p[None, :], thr)[0]
        assert np.array_equal(got, subsets[best]), (p, thr, got, subsets[best])


def check_cdf_invariants(cdf_keep, seed=5):
    """On larger random rows: kept mass > thr, and dropping the lightest kept block
    leaves mass <= thr (up to fp64 rounding); thr = 1 keeps everything."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(200, 0.5), size=30)
    for thr in (0.3, 0.8, 0.9, 0.99):
        keep = cdf_keep(p, thr)
        kept_mass = np.where(keep, p, 0).sum(-1)
        lightest = np.where(keep, p, np.inf).min(-1)
        assert np.all(kept_mass >= thr - 1e-12)
        assert np.all(kept_mass - lightest <= thr + 1e-12)
    assert cdf_keep(p, 1.0).all()


# ------------------------------------------------------------------ a5 STA
def check_sta_golden(sta_mask):
    for case in load_sta_windows():
        got = sta_mask(*case["grid"], *case["half"])
        assert np.array_equal(got, case["mask"]), case["grid"]


def check_sta_counts(sta_mask):
    """Closed form: row count = product over axes of the clipped window lengths;
    the mask is symmetric; the diagonal is always kept."""
    T, H, W, wt, wh, ww = 5, 4, 6, 1, 2, 0
    m = sta_mask(T, H, W, wt, wh, ww)
    assert np.array_equal(m, m.T) and np.all(np.diag(m) == 1)
    for i in range(T * H * W):
        t, y, x = i // (H * W), (i // W) % H, i % W
        n = ((min(T - 1, t + wt) - max(0, t - wt) + 1) * (min(H - 1, y + wh) - max(0, y - wh) + 1)
             * (min(W - 1, x + ww) - max(0, x - ww) + 1))
        assert m[i].sum() == n


# ------------------------------------------------------------------ a6 CSR
def check_csr(csr_from_mask, seed=6):
    """kv_nb is the row popcount; the first kv_nb indices are the kept blocks,
    strictly ascending ([P1] BlockMask creation; ascending order by reading)."""
    rng = np.random.default_rng(seed)
    mask = rng.random((2, 3, 17, 17)) < 0.4
    mask[0, 0, 0] = False
    mask[0, 0, 1] = True
    kv_nb, kv_inds = csr_from_mask(mask)
    assert kv_nb.dtype == np.int32 and kv_inds.dtype == np.int32
    for idx in np.ndindex(mask.shape[:-1]):
        want = np.nonzero(mask[idx])[0]
        assert kv_nb[idx] == len(want)
        assert np.array_equal(kv_inds[idx][:len(want)], want)


# ------------------------------------------------------------------ whole builder
def torch_nabla_mask(q, k, sta, thr):
    """An independent float64 torch statement of the page's nablaT_v2 procedure
    ([P1]): head-major view, 64-token means, pooled product over sqrt(D), softmax,
    ascending stable sort, running sum, >= 1 - thr, flags scattered back to block
    order, OR with the STA window, row counts."""
    qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float64)).permute(0, 2, 1, 3)
    kt = torch.from_numpy(np.ascontiguousarray(k, dtype=np.float64)).permute(0, 2, 1, 3)
    B, h, S, D = qt.shape
    n = S // 64
    qm = qt.reshape(B, h, n, 64, D).mean(3)
    km = kt.reshape(B, h, n, 64, D).mean(3)
    prob = torch.softmax(torch.einsum("bhid,bhjd->bhij", qm, km) / math.sqrt(D), -1)
    vals, order = torch.sort(prob, dim=-1, stable=True)
    run = torch.cumsum(vals, -1)
    flags = torch.zeros_like(prob, dtype=torch.bool)
    flags.scatter_(-1, order, run >= (1.0 - thr))
    full = flags | torch.from_numpy(np.asarray(sta, dtype=bool))[None, None]
    return full.sum(-1).to(torch.int32).numpy(), full.numpy(), prob.numpy()


def check_builder_vs_torch(build_mask, q, k, sta, thr):
    got = build_mask(q, k, sta, thr)
    nb, full, prob = torch_nabla_mask(q, k, sta, thr)
    assert np.allclose(got["p"], prob, rtol=0, atol=1e-14)
    near = np.abs(got["c"] - (1.0 - thr)) < 1e-12
    assert np.array_equal(got["mask"][~near], full[~near])
    if not near.any():
        assert np.array_equal(got["kv_nb"], nb)


def check_sta_forced(build_mask, q, k, s1, seed=7):
    """STA blocks are always kept; an all-ones STA keeps everything ([P1] OR;
    [P4] Hybrid Integration, M = M_nabla OR M_STA)."""
    rng = np.random.default_rng(seed)
    sta = (rng.random((s1, s1)) < 0.3).astype(np.uint8)
    got = build_mask(q, k, sta, 0.5)
    assert np.all(got["mask"][:, :, sta.astype(bool)])
    full = build_mask(q, k, np.ones((s1, s1), np.uint8), 0.5)
    assert full["mask"].all()
    allthr = build_mask(q, k, np.zeros((s1, s1), np.uint8), 1.0)
    assert allthr["mask"].all()


# ------------------------------------------------------------------ a7 attention
def sdpa64(q, k, v, scale, token_mask=None):
    """torch fp64 scaled_dot_product_attention on [B, S, h, D] numpy inputs."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).permute(0, 2, 1, 3)
    am = None if token_mask is None else torch.from_numpy(token_mask)
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=am,
                                                         scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def check_attention_dense(block_sparse_attention, csr_from_mask, seed=8):
    """A full mask equals unmasked dense attention (torch fp64 SDPA)."""
    rng = np.random.default_rng(seed)
    B, S, h, D = 1, 256, 2, 32
    q, k, v = (rng.standard_normal((B, S, h, D)) for _ in range(3))
    nb, inds = csr_from_mask(np.ones((B, h, 4, 4), bool))
    got = block_sparse_attention(q, k, v, nb, inds, 0.3)
    assert np.allclose(got, sdpa64(q, k, v, 0.3), rtol=0, atol=1e-12)


def check_attention_masked(block_sparse_attention, csr_from_mask, seed=9):
    """A random block mask equals token-masked dense attention (torch fp64 SDPA with
    a boolean mask expanded from 64x64 blocks, [P4] Expansion); empty rows give 0."""
    rng = np.random.default_rng(seed)
    B, S, h, D = 2, 384, 2, 16
    s1 = S // 64
    q, k, v = (rng.standard_normal((B, S, h, D)) for _ in range(3))
    mask = rng.random((B, h, s1, s1)) < 0.5
    mask[0, 1, 3] = False  # one empty row
    mask[1, 0, 2] = False
    mask[1, 0, 2, 5] = True  # one single-block row
    nb, inds = csr_from_mask(mask)
    got = block_sparse_attention(q, k, v, nb, inds, 1.0 / math.sqrt(D))
    tok = np.repeat(np.repeat(mask, 64, axis=2), 64, axis=3)
    want = sdpa64(q, k, v, 1.0 / math.sqrt(D), tok)
    rows_empty = ~mask.any(-1)
    for b, hh, i in zip(*np.nonzero(rows_empty)):
        want[b, i * 64:(i + 1) * 64, hh] = 0.0
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def check_attention_closed_form(block_sparse_attention, csr_from_mask):
    """Closed forms: (1) constant v gives that constant; (2) q = a*e0 and keys of
    block j all equal b_j*e0, v of block j all equal c_j: weights are
    exp(scale*a*b_j) per kept block, so o = sum w_j c_j / sum w_j."""
    B, S, h, D = 1, 192, 1, 4
    s1 = 3
    q = np.zeros((B, S, h, D))
    k = np.zeros((B, S, h, D))
    v = np.full((B, S, h, D), 0.7)
    mask = np.array([[[[1, 0, 1], [0, 1, 0], [1, 1, 1]]]], bool)
    nb, inds = csr_from_mask(mask)
    assert np.allclose(block_sparse_attention(q, k, v, nb, inds, 0.5), 0.7, atol=1e-15)
    a, bj, cj = 2.0, np.array([0.5, -1.0, 1.5]), np.array([1.0, 2.0, 4.0])
    q[..., 0] = a
    for j in range(s1):
        k[0, 64 * j:64 * (j + 1), 0, 0] = bj[j]
        v[0, 64 * j:64 * (j + 1), 0, :] = cj[j]
    scale = 0.25
    got = block_sparse_attention(q, k, v, nb, inds, scale)
    for i in range(s1):
        keep = mask[0, 0, i]
        w = np.exp(scale * a * bj) * keep
        want = (w * cj).sum() / w.sum()
        assert np.allclose(got[0, 64 * i:64 * (i + 1), 0, :], want, rtol=1e-14, atol=0)
