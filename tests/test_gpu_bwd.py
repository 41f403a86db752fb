"""Attention backward on the GPU vs the fp64 oracle, through the C ABI.

The mask comes from the GPU mask builder and o from the GPU forward (what a
training step stores); the oracle gets the same mask and the same o (reading
R17).  Tolerances, derived from the arithmetic (the pages fix none for the
backward): fp32 storage, max|err| <= 1e-4 * max|ref| per gradient (fp32 sums
of up to ~10^5 terms); bf16 storage, P and dz are rounded to bf16 before the
tensor-core products (as the forward rounds P, reading R9) and the gradients
are rounded to bf16: dz sums to zero along a row, so dq and dk are sums with
cancellation and carry about 2^-8 of relative error on average:
max|err| <= 2e-2 * max|ref| and mean|err| <= 5e-3 * mean|ref|.  At full size the checks are the invariants
sum_u dk_u = 0 and sum_u dv_u = sum of dout over rows that keep something,
plus exact oracle values on sampled blocks.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_nablat_gb300 import workloads as W
from oracle import nabla_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"f32": (1e-4, None), "bf16": (2e-2, 5e-3)}


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


def run_gpu(nabla, w, data, dout, thr=None, nb=None, inds=None):
    q, k, v = (nabla.from_storage(data[n], DEV) for n in "qkv")
    g = nabla.from_storage(dout, DEV)
    if nb is None:
        sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=DEV)
        nb, inds = nabla.nabla_build_mask(q, k, sta, w.thr[0] if thr is None else thr)
    else:
        nb, inds = torch.from_numpy(nb).to(DEV), torch.from_numpy(inds).to(DEV)
    o = nabla.nabla_attn_fwd(q, k, v, nb, inds, w.scale)
    dq, dk, dv = nabla.nabla_attn_bwd(q, k, v, o, g, nb, inds, w.scale)
    torch.cuda.synchronize()
    status = nabla.nabla_get_last_device_status()
    to_np = lambda t: t.float().cpu().numpy()  # noqa: E731
    return (to_np(dq), to_np(dk), to_np(dv), to_np(o), nb.cpu().numpy(), inds.cpu().numpy(),
            status)


def compare(w, got, ref):
    amax, amean = TOL[w.dtype]
    out = []
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        err = np.abs(g - r)
        scale = np.abs(r).max()
        assert err.max() <= amax * scale, (name, err.max(), scale)
        if amean is not None:
            assert err.mean() <= amean * np.abs(r).mean(), (name, err.mean(), np.abs(r).mean())
        out.append((float(err.max() / scale), float(err.mean() / np.abs(r).mean())))
    return out


def full_check(nabla, w, seed=0, thr=None, nb=None, inds=None):
    data = W.generate(w, seed)
    dout = W.generate_dout(w, seed)
    dq, dk, dv, o, nb, inds, status = run_gpu(nabla, w, data, dout, thr, nb, inds)
    assert status == 0
    qf, kf, vf, gf = (W.as_float(x) for x in (data["q"], data["k"], data["v"], dout))
    ref = O.block_sparse_attention_bwd(qf, kf, vf, gf, nb, inds, w.scale, o=o)
    return compare(w, (dq, dk, dv), ref), (dq, dk, dv, nb, inds, gf)


@pytest.mark.parametrize("name", ["tiny_f32", "small_bf16"])
def test_bwd_small_configs(nabla, name):
    rel, _ = full_check(nabla, W.WORKLOADS[name])
    print("BWD", name, "(max err / max |ref|, mean err / mean |ref|) for dq, dk, dv:", rel)


@pytest.mark.parametrize("B,h,D,s1,dtype", [(2, 3, 64, 37, "bf16"), (1, 2, 128, 10, "f32"),
                                            (1, 2, 64, 24, "f32")])
def test_bwd_ragged_and_head_dims(nabla, B, h, D, s1, dtype):
    w = W.custom(f"bwd{s1}", B, h, D, 64 * s1, (s1, 1, 1), sigma=0.75, rho=0.8, thr=(0.7,),
                 dtype=dtype)
    rel, _ = full_check(nabla, w, seed=3)
    print("BWD", w.name, rel)


def test_bwd_empty_rows_and_unkept_key_blocks(nabla):
    """Query blocks that keep nothing get dq = 0 and add nothing; key blocks
    that nobody keeps get dk = dv = 0."""
    w = W.custom("bwd_empty", 1, 2, 64, 64 * 8, (8, 1, 1), dtype="f32")
    rng = np.random.default_rng(7)
    keep = rng.random((1, 2, 8, 8)) < 0.5
    keep[0, 0, 2] = False          # an empty query block
    keep[0, 1, :, 5] = False       # key block 5 of head 1 kept by nobody
    keep[0, 1, 0, 1] = True
    nb, inds = O.csr_from_mask(keep)
    rel, (dq, dk, dv, *_rest) = full_check(nabla, w, seed=4, nb=nb, inds=inds)
    assert np.all(dq[0, 128:192, 0] == 0.0)
    assert np.all(dk[0, 320:384, 1] == 0.0) and np.all(dv[0, 320:384, 1] == 0.0)


def test_bwd_480p_invariants_and_sampled_blocks(nabla):
    w = W.WORKLOADS["480p_bf16"]
    data = W.generate(w, 0)
    dout = W.generate_dout(w, 0)
    dq, dk, dv, o, nb, inds, status = run_gpu(nabla, w, data, dout)
    assert status == 0
    gf = W.as_float(dout)
    for hh in range(w.h):
        # sum over key tokens of dk vanishes; sum of dv equals sum of dout over kept rows
        sk = dk[0, :, hh].astype(np.float64).sum(axis=0)
        assert np.abs(sk).max() <= 2e-2 * np.abs(dk[0, :, hh]).sum(axis=0).max()
        kept_rows = np.repeat(nb[0, hh] > 0, 64)
        sv = dv[0, :, hh].astype(np.float64).sum(axis=0)
        want = gf[0, kept_rows, hh].astype(np.float64).sum(axis=0)
        assert np.abs(sv - want).max() <= 2e-2 * np.abs(gf[0, :, hh]).sum(axis=0).max()
    qf, kf, vf = (W.as_float(data[n]) for n in "qkv")
    rng = np.random.default_rng(9)
    qbl = sorted({(0, int(rng.integers(w.h)), int(rng.integers(w.s1))) for _ in range(6)})
    rdq, _, _ = O.block_sparse_attention_bwd(qf, kf, vf, gf, nb, inds, w.scale, o=o, qblocks=qbl)
    amax, amean = TOL[w.dtype]
    for b, hh, i in qbl:
        r, g = rdq[b, 64 * i:64 * i + 64, hh], dq[b, 64 * i:64 * i + 64, hh]
        assert np.abs(g - r).max() <= amax * np.abs(r).max()
    # one key block: every query block that kept it
    hh, j = 5, 77
    users = [(0, hh, i) for i in range(w.s1) if j in set(inds[0, hh, i, :nb[0, hh, i]].tolist())]
    _, rdk, rdv = O.block_sparse_attention_bwd(qf, kf, vf, gf, nb, inds, w.scale, o=o,
                                               qblocks=users)
    for g, r in ((dk, rdk), (dv, rdv)):
        r, g = r[0, 64 * j:64 * j + 64, hh], g[0, 64 * j:64 * j + 64, hh]
        assert np.abs(g - r).max() <= amax * np.abs(r).max()
        assert np.abs(g - r).mean() <= amean * np.abs(r).mean()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_bad_index_is_reported_and_skipped(nabla, dtype):
    w = W.custom("bwd_bad", 1, 1, 64, 64 * 4, (4, 1, 1), dtype=dtype)
    keep = np.ones((1, 1, 4, 4), bool)
    nb, inds = O.csr_from_mask(keep)
    inds[0, 0, 1, 2] = 9           # out of range: skipped
    data = W.generate(w, 5)
    dout = W.generate_dout(w, 5)
    dq, dk, dv, o, *_rest, status = run_gpu(nabla, w, data, dout, nb=nb, inds=inds)
    assert status == 5  # NABLA_ERR_BAD_INDEX
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


@pytest.mark.parametrize("name", ["small_bf16", "tiny_f32"])
def test_forward_lse_matches_oracle_and_feeds_the_backward(nabla, name):
    """nabla_attn_fwd_lse: the same o as nabla_attn_fwd (bit for bit), the rows'
    base-2 log-sum-exp within 1e-5 (absolute, on values of order 10), and a
    backward given that lse equal to one that computes its own."""
    w = W.WORKLOADS[name]
    data = W.generate(w, 0)
    dout = W.generate_dout(w, 0)
    q, k, v = (nabla.from_storage(data[n], DEV) for n in "qkv")
    g = nabla.from_storage(dout, DEV)
    sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=DEV)
    nb, inds = nabla.nabla_build_mask(q, k, sta, w.thr[0])
    o = nabla.nabla_attn_fwd(q, k, v, nb, inds, w.scale)
    o2, lse = nabla.nabla_attn_fwd_lse(q, k, v, nb, inds, w.scale)
    assert torch.equal(o, o2)
    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    ref = O.attention_lse2(qf, kf, nb.cpu().numpy(), inds.cpu().numpy(), w.scale)
    got = lse.cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got))
    assert np.abs(got[fin] - ref[fin]).max() <= 1e-5 * max(1.0, np.abs(ref[fin]).max())
    a = nabla.nabla_attn_bwd(q, k, v, o, g, nb, inds, w.scale)
    b = nabla.nabla_attn_bwd(q, k, v, o, g, nb, inds, w.scale, lse=lse)
    assert nabla.nabla_get_last_device_status() == 0
    for x, y in zip(a, b):
        xf, yf = x.float(), y.float()
        assert (xf - yf).abs().max().item() <= 1e-2 * xf.abs().max().item()


def test_bwd_bf16_empty_rows_and_unkept_key_blocks(nabla):
    """The tensor-core path: a query block that keeps nothing gets dq = 0, a key
    block that nobody keeps gets dk = dv = 0, odd block count (a pair half past
    the end)."""
    w = W.custom("bwd_empty_bf16", 1, 2, 128, 64 * 9, (9, 1, 1), dtype="bf16")
    rng = np.random.default_rng(8)
    keep = rng.random((1, 2, 9, 9)) < 0.5
    keep[0, 0, 2] = False
    keep[0, 1, :, 5] = False
    keep[0, 1, 0, 1] = True
    nb, inds = O.csr_from_mask(keep)
    rel, (dq, dk, dv, *_rest) = full_check(nabla, w, seed=4, nb=nb, inds=inds)
    assert np.all(dq[0, 128:192, 0] == 0.0)
    assert np.all(dk[0, 320:384, 1] == 0.0) and np.all(dv[0, 320:384, 1] == 0.0)
    print("BWD", w.name, rel)
