"""Pins of the oracle's attention backward (CPU, no GPU).

Source: gist.science NABLA summary, "Dual-Phase Acceleration" and Experimental
Results (pre-training with NABLA): the backward is the gradient of the block-
sparse attention of a7.  None of these tests reuses the oracle's formulas:
  * central finite differences of the loss sum(dout * o), with o from the
    oracle's forward (pinned on its own against torch SDPA);
  * torch autograd through scaled_dot_product_attention with the expanded
    token mask;
  * invariants that hold for any input: sum_u dk_u = 0 (the dz of a row sums
    to zero) and sum_u dv_u = sum of dout over rows that keep something;
  * a closed form: identical v rows make o independent of the scores, so dq
    and dk vanish.
"""
import numpy as np
import pytest

from oracle import nabla_oracle as O

BLOCK = 64


def _csr(rows):
    """rows: per (b, h) a list of per-query-block kept lists -> (kv_nb, kv_inds)."""
    B, h, s1 = len(rows), len(rows[0]), len(rows[0][0])
    nb = np.zeros((B, h, s1), np.int32)
    inds = np.full((B, h, s1, s1), -1, np.int32)
    for b in range(B):
        for hh in range(h):
            for i, lst in enumerate(rows[b][hh]):
                nb[b, hh, i] = len(lst)
                inds[b, hh, i, :len(lst)] = sorted(lst)
    return nb, inds


def _random_csr(rng, B, h, s1, p_keep=0.5, allow_empty=True):
    rows = []
    for _ in range(B):
        per_h = []
        for _ in range(h):
            lst = []
            for i in range(s1):
                keep = [j for j in range(s1) if rng.random() < p_keep]
                if not keep and not allow_empty:
                    keep = [int(rng.integers(s1))]
                lst.append(keep)
            per_h.append(lst)
        rows.append(per_h)
    return _csr(rows)


def _loss(q, k, v, dout, nb, inds, scale):
    o = O.block_sparse_attention(q, k, v, nb, inds, scale)
    return float((dout * o).sum())


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(0)
    B, h, D, s1 = 1, 2, 4, 3
    S = s1 * BLOCK
    q, k, v, dout = (rng.standard_normal((B, S, h, D)) for _ in range(4))
    # head 0: block 1 keeps nothing (its rows contribute nothing); head 1: all rows keep
    nb, inds = _csr([[[[0, 2], [], [0, 1, 2]], [[1], [0, 2], [2]]]])
    scale = 0.7
    dq, dk, dv = O.block_sparse_attention_bwd(q, k, v, dout, nb, inds, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        idx = [tuple(int(rng.integers(n)) for n in x.shape) for _ in range(40)]
        idx += [(0, 64 + 5, 0, 1)]  # a row of the empty query block (head 0)
        for ix in idx:
            xp, xm = x.copy(), x.copy()
            xp[ix] += eps
            xm[ix] -= eps
            args = {"q": q, "k": k, "v": v}
            fp = _loss(*(xp if n == name else args[n] for n in "qkv"), dout, nb, inds, scale)
            fm = _loss(*(xm if n == name else args[n] for n in "qkv"), dout, nb, inds, scale)
            fd = (fp - fm) / (2 * eps)
            assert abs(fd - g[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix, fd, g[ix])
    assert np.all(dq[0, 64:128, 0] == 0.0)  # the empty block's rows get no gradient


def test_backward_matches_torch_autograd_sdpa():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    B, h, D, s1 = 2, 2, 16, 6
    S = s1 * BLOCK
    q, k, v, dout = (rng.standard_normal((B, S, h, D)) for _ in range(4))
    nb, inds = _random_csr(rng, B, h, s1, 0.45, allow_empty=False)
    scale = 1.0 / np.sqrt(D)
    mask = np.zeros((B, h, S, S), bool)
    for b in range(B):
        for hh in range(h):
            for i in range(s1):
                for j in inds[b, hh, i, :nb[b, hh, i]]:
                    mask[b, hh, i * BLOCK:(i + 1) * BLOCK, j * BLOCK:(j + 1) * BLOCK] = True
    tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.tensor(mask), scale=scale)
    to.backward(torch.tensor(dout.transpose(0, 2, 1, 3)))
    ref = [t.grad.numpy().transpose(0, 2, 1, 3) for t in (tq, tk, tv)]
    got = O.block_sparse_attention_bwd(q, k, v, dout, nb, inds, scale)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, rtol=1e-9, atol=1e-11)


def test_backward_invariants_and_stored_output():
    rng = np.random.default_rng(2)
    B, h, D, s1 = 1, 3, 8, 7
    S = s1 * BLOCK
    q, k, v, dout = (rng.standard_normal((B, S, h, D)) for _ in range(4))
    nb, inds = _random_csr(rng, B, h, s1, 0.4, allow_empty=True)
    nb[0, 1, 3] = 0
    scale = 0.3
    dq, dk, dv = O.block_sparse_attention_bwd(q, k, v, dout, nb, inds, scale)
    for hh in range(h):
        np.testing.assert_allclose(dk[0, :, hh].sum(axis=0), 0.0, atol=1e-11)
        kept_rows = np.repeat(nb[0, hh] > 0, BLOCK)
        np.testing.assert_allclose(dv[0, :, hh].sum(axis=0),
                                   dout[0, kept_rows, hh].sum(axis=0), atol=1e-11)
    # R17: the exact stored output gives the same gradients
    o = O.block_sparse_attention(q, k, v, nb, inds, scale)
    for a, b in zip((dq, dk, dv), O.block_sparse_attention_bwd(q, k, v, dout, nb, inds, scale,
                                                               o=o)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_backward_identical_values_kill_query_and_key_gradients():
    rng = np.random.default_rng(3)
    B, h, D, s1 = 1, 2, 8, 4
    S = s1 * BLOCK
    q, k, dout = (rng.standard_normal((B, S, h, D)) for _ in range(3))
    v = np.broadcast_to(rng.standard_normal((1, 1, h, D)), (B, S, h, D)).copy()
    nb, inds = _random_csr(rng, B, h, s1, 0.6, allow_empty=False)
    dq, dk, dv = O.block_sparse_attention_bwd(q, k, v, dout, nb, inds, 0.5)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


def test_lse_closed_form_and_identity():
    rng = np.random.default_rng(6)
    B, h, D, s1 = 1, 2, 8, 5
    S = s1 * BLOCK
    q, k, v = (rng.standard_normal((B, S, h, D)) for _ in range(3))
    nb, inds = _random_csr(rng, B, h, s1, 0.5, allow_empty=True)
    nb[0, 0, 1] = 0
    # q = 0: every score is 0, so the sum is the number of kept tokens
    lz = O.attention_lse2(np.zeros_like(q), k, nb, inds, 0.4)
    for hh in range(h):
        for i in range(s1):
            got = lz[0, hh, 64 * i:64 * i + 64]
            if nb[0, hh, i] == 0:
                assert np.all(got == -np.inf)
            else:
                np.testing.assert_allclose(got, np.log2(64.0 * nb[0, hh, i]), rtol=1e-14)
    # 2^(z log2(e) - lse2) are the softmax weights: they rebuild the forward's o
    scale = 0.4
    lse = O.attention_lse2(q, k, nb, inds, scale)
    o = O.block_sparse_attention(q, k, v, nb, inds, scale)
    for hh in range(h):
        for i in range(s1):
            n = nb[0, hh, i]
            if n == 0:
                continue
            tok = (inds[0, hh, i, :n][:, None] * 64 + np.arange(64)[None, :]).ravel()
            rows = slice(64 * i, 64 * i + 64)
            z = scale * q[0, rows, hh] @ k[0, tok, hh].T
            w = np.exp2(z / np.log(2.0) - lse[0, hh, rows][:, None])
            np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-12)
            np.testing.assert_allclose(w @ v[0, tok, hh], o[0, rows, hh], rtol=1e-10, atol=1e-12)
