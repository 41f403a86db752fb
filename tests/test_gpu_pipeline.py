"""The widened rows working together on the GPU, against the oracle.

* fractal order -> mask build -> attention -> inverse order: a raster latent
  goes through the whole layer, and the result equals the oracle applied to
  the oracle's own fractal flattening of the same latent;
* the top-k selector's CSR drives the attention forward directly.
"""
import numpy as np
import pytest
import torch

import mask_tolerance as MT
from block_sparse_attention_nablat_gb300 import workloads as W
from oracle import nabla_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def nabla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    from block_sparse_attention_nablat_gb300 import nabla as N

    try:
        N.load()
    except RuntimeError:
        __graft_entry__.build()
        N.load()
    return N


def _mask_of(nb, inds, s1):
    m = np.zeros(nb.shape + (s1,), bool)
    for idx in np.ndindex(nb.shape):
        m[idx][inds[idx][:nb[idx]]] = True
    return m


def test_raster_layer_through_fractal_order(nabla):
    """T=4 frames of 16x16 tokens, P=8: 16 blocks of one 8x8 patch each."""
    w = W.custom("layer", 1, 2, 64, 4 * 16 * 16, (4, 2, 2), sigma=0.75, rho=0.8, thr=(0.8,))
    data = W.generate(w, 2)  # drawn in fractal order; reinterpret the token axis as raster
    T, H, Wd = 4, 16, 16
    raster = {n: W.as_float(data[n]).reshape(1, T, H, Wd, w.h, w.D) for n in "qkv"}
    dev = {n: torch.from_numpy(np.ascontiguousarray(raster[n])).to(DEV) for n in "qkv"}
    flat = {n: nabla.nabla_fractal_flatten(dev[n], 8) for n in "qkv"}
    sta = nabla.nabla_sta_mask(*w.grid, 1, 1, 1, device=DEV)
    nb, inds = nabla.nabla_build_mask(flat["q"], flat["k"], sta, 0.8)
    o = nabla.nabla_attn_fwd(flat["q"], flat["k"], flat["v"], nb, inds, w.scale)
    back = nabla.nabla_fractal_unflatten(o, T, H, Wd, 8)
    assert nabla.nabla_get_last_device_status() == 0
    # oracle: its own flattening, mask and attention, then its own inverse
    of = {n: O.fractal_flatten(raster[n].astype(np.float64), 8) for n in "qkv"}
    ref = O.build_mask(of["q"], of["k"], O.sta_mask(*w.grid, 1, 1, 1), 0.8)
    nbh, indh = nb.cpu().numpy(), inds.cpu().numpy()
    got = _mask_of(nbh, indh, w.s1)
    sta_h = O.sta_mask(*w.grid, 1, 1, 1)
    theta = MT.block_margins(of["q"], of["k"], ref["p"])
    amb = O.ambiguous_blocks(ref["c"], ref["t"], sta_h) | MT.near_tie_blocks(
        ref["p"], ref["cdf_mask"], theta, sta_h)
    assert np.array_equal(got[~amb], ref["mask"][~amb])
    oref = O.block_sparse_attention(of["q"], of["k"], of["v"], nbh, indh, w.scale)
    want = O.fractal_unflatten(oref, T, H, Wd, 8)
    assert np.abs(back.cpu().numpy() - want).max() <= 1e-5


def test_topk_mask_drives_attention(nabla):
    w = W.WORKLOADS["small_bf16"]
    data = W.generate(w, 4)
    q, k, v = (nabla.from_storage(data[n], DEV) for n in "qkv")
    nb, inds = nabla.nabla_build_mask_topk(q, k, 0.25)
    o = nabla.nabla_attn_fwd(q, k, v, nb, inds, w.scale)
    assert nabla.nabla_get_last_device_status() == 0
    nbh, indh = nb.cpu().numpy(), inds.cpu().numpy()
    assert np.all(nbh == 32)
    qf, kf, vf = (W.as_float(data[n]) for n in "qkv")
    ref = O.block_sparse_attention(qf, kf, vf, nbh, indh, w.scale)
    err = np.abs(o.float().cpu().numpy() - ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
