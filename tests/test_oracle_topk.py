"""Pins of the oracle's top-k block selector (CPU, no GPU).

Source: FastVideo API reference, attention backends index, sla.get_block_map
(smooth-k, 64-token mean pooling of q and the smoothed k, plain pooled product,
topk = min(K, int(topk_ratio * K)) largest per query block); reading R14 for
ties (the kept set is the last k of the ascending (score, index) order).
"""
import numpy as np
import pytest

from oracle import nabla_oracle as O


def _const_blocks(means):
    """[B, h, s1, D] block means -> [B, S, h, D] tokens equal to their block's mean."""
    B, h, s1, D = means.shape
    return np.repeat(np.transpose(means, (0, 2, 1, 3))[:, :, None], 64, axis=2).reshape(
        B, s1 * 64, h, D)


def test_topk_hand_worked_rows():
    # q blocks all (1, 0); k block means (b_j, 0) with b = [3, 1, 4, 1]: smooth-k
    # subtracts mean(b) = 2.25, so every row scores [0.75, -1.25, 1.75, -1.25].
    qm = np.zeros((1, 1, 4, 2)); qm[..., 0] = 1.0
    km = np.zeros((1, 1, 4, 2)); km[..., 0] = [3, 1, 4, 1]
    q, k = _const_blocks(qm), _const_blocks(km)
    r = O.topk_mask(q, k, 0.5)           # k = 2: blocks 2 and 0
    assert r["topk"] == 2
    assert np.allclose(r["scores"][0, 0, 0], [0.75, -1.25, 1.75, -1.25])
    assert r["kv_inds"][0, 0, 0, :2].tolist() == [0, 2]
    r = O.topk_mask(q, k, 0.75)          # k = 3: the tie between blocks 1 and 3 keeps 3
    assert r["kv_inds"][0, 0, 0, :3].tolist() == [0, 2, 3]
    r = O.topk_mask(q, k, 0.7)           # int(2.8) = 2, not a rounded 3
    assert r["topk"] == 2
    r = O.topk_mask(q, k, 0.2)           # int(0.8) = 0: nothing kept
    assert r["topk"] == 0 and np.all(r["kv_nb"] == 0)
    r = O.topk_mask(q, k, 1.0)
    assert np.all(r["kv_nb"] == 4)


def test_topk_brute_force_order():
    rng = np.random.default_rng(3)
    q = rng.integers(-2, 3, size=(1, 64 * 10, 2, 4)).astype(np.float64)
    k = rng.integers(-2, 3, size=(1, 64 * 10, 2, 4)).astype(np.float64)
    for ratio in (0.1, 0.35, 0.5, 0.99):
        r = O.topk_mask(q, k, ratio)
        sc, keep, kk = r["scores"], r["mask"], r["topk"]
        assert np.all(keep.sum(-1) == kk)
        for idx in np.ndindex(sc.shape[:-1]):
            s, m = sc[idx], keep[idx]
            for a in np.nonzero(m)[0]:          # every kept block outranks every dropped one
                for b in np.nonzero(~m)[0]:
                    assert s[a] > s[b] or (s[a] == s[b] and a > b)


def test_topk_smooth_k_does_not_change_the_selection():
    """Subtracting the sequence mean of k shifts every score of a row by one
    constant, so the selection equals top-k of the plain pooled product."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((2, 64 * 12, 3, 8))
    k = rng.standard_normal((2, 64 * 12, 3, 8)) + 5.0  # a large mean to smooth away
    r = O.topk_mask(q, k, 0.4)
    plain = np.matmul(O.pool_blocks(q), np.swapaxes(O.pool_blocks(k), -1, -2))
    order = np.argsort(plain, axis=-1, kind="stable")
    keep = np.zeros(plain.shape, bool)
    np.put_along_axis(keep, order[..., -r["topk"]:], True, axis=-1)
    assert np.array_equal(keep, r["mask"])
