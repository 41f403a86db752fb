"""Pins of the oracle's fractal flatten / unflatten (CPU, no GPU).

The order itself is pinned by hand-derived fixtures (tests/golden/fractal_order.txt);
the rest are properties any correct implementation has: it is a permutation, the
inverse undoes it, each 64-token block of the output is one 8 x 8 patch of one
frame, P = 1 is the identity.
"""
import os

import numpy as np
import pytest

from oracle import nabla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fractal_order.txt")


def _cases():
    cases, shape = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("shape:"):
            shape = tuple(int(v) for v in line.split()[1:])
        elif line.startswith("order:"):
            cases.append((shape, [int(v) for v in line.split()[1:]]))
    return cases


@pytest.mark.parametrize("shape,order", _cases())
def test_fractal_golden(shape, order):
    T, H, W, P = shape
    x = np.arange(T * H * W).reshape(1, T, H, W, 1, 1)
    y = O.fractal_flatten(x, P).ravel()
    assert y.tolist() == order


def test_fractal_roundtrip_and_permutation():
    rng = np.random.default_rng(1)
    for (T, H, W, P) in [(3, 16, 24, 8), (2, 8, 8, 4), (1, 6, 10, 2), (4, 5, 7, 1)]:
        x = rng.standard_normal((2, T, H, W, 3, 4))
        y = O.fractal_flatten(x, P)
        assert y.shape == (2, T * H * W, 3, 4)
        assert sorted(y.ravel().tolist()) == sorted(x.ravel().tolist())
        assert np.array_equal(O.fractal_unflatten(y, T, H, W, P), x)


def test_fractal_blocks_are_patches():
    """With P = 8 every 64-token block holds exactly one 8 x 8 patch of one frame."""
    T, H, W = 2, 16, 24
    t, yy, xx = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    coords = np.stack([t, yy, xx], -1).reshape(1, T, H, W, 1, 3)
    f = O.fractal_flatten(coords, 8).reshape(T * H * W // 64, 64, 3)
    for blk in f:
        assert len(set(blk[:, 0])) == 1                       # one frame
        assert blk[:, 1].max() - blk[:, 1].min() == 7          # 8 rows
        assert blk[:, 2].max() - blk[:, 2].min() == 7          # 8 columns
        assert blk[:, 1].min() % 8 == 0 and blk[:, 2].min() % 8 == 0
        assert len({(a, b) for _, a, b in blk}) == 64
    # frames stay in time order: block b belongs to frame b // (H*W/64)
    assert [int(b[0, 0]) for b in f] == [i // (H * W // 64) for i in range(len(f))]


def test_fractal_patch_size_one_is_identity():
    x = np.arange(2 * 3 * 5 * 2).reshape(1, 2, 3, 5, 2, 1)
    assert np.array_equal(O.fractal_flatten(x, 1), x.reshape(1, 30, 2, 1))


def test_fractal_rejects_ragged_patches():
    with pytest.raises(ValueError):
        O.fractal_flatten(np.zeros((1, 1, 6, 8, 1, 1)), 4)
