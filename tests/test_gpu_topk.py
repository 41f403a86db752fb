"""Top-k block selector (sla.get_block_map) on the GPU vs the fp64 oracle.

The CUDA path ranks the rows of the fp32 pooled map <qa_i, ka_j> / sqrt(D),
while the oracle ranks the fp64 smooth-k scores <qa_i, ka_j - mean_j ka_j>;
the two orders agree in exact arithmetic (a per-row shift and a positive
scale).  Tolerance: every row keeps exactly topk blocks, and a block may differ
from the oracle only if its oracle score lies within TIE_REL * ||qa_i|| *
max_j ||ka_j|| of the row's topk-th score (an order float32 cannot resolve),
at most 0.1% of the entries.  Designed inputs whose scores are exact in
float32 must match bit for bit (ties included).
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_nablat_gb300 import workloads as W
from oracle import nabla_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIE_REL = 2e-5
MAX_MISMATCH_FRAC = 1e-3


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


def to_mask(nb, inds, s1):
    """Boolean mask of the kept prefix; checks that the prefix ascends strictly."""
    pos = np.arange(s1)
    valid = pos < nb[..., None]
    sel = np.where(valid, inds, s1).astype(np.int64)
    assert np.all((sel >= 0) & (sel <= s1))
    d = np.diff(np.where(valid, inds, np.iinfo(np.int32).max).astype(np.int64), axis=-1)
    assert np.all(d[valid[..., 1:]] > 0), "kv_inds prefix not strictly ascending"
    m = np.zeros(nb.shape + (s1 + 1,), dtype=bool)
    np.put_along_axis(m, sel, True, axis=-1)
    return m[..., :s1]


def gpu_topk(nabla, q, k, ratio):
    nb, inds = nabla.nabla_build_mask_topk(q, k, ratio)
    assert nabla.nabla_get_last_device_status() == 0
    return nb.cpu().numpy(), inds.cpu().numpy()


def check_topk(qf, kf, nb, inds, ratio):
    ref = O.topk_mask(qf, kf, ratio)
    s1 = ref["scores"].shape[-1]
    kk = ref["topk"]
    assert np.all(nb == kk)
    got = to_mask(nb, inds, s1)
    mism = got != ref["mask"]
    if kk in (0, s1):
        assert not mism.any()
        return 0
    sc = ref["scores"]
    order = np.argsort(sc, axis=-1, kind="stable")
    kth = np.take_along_axis(sc, order[..., s1 - kk:s1 - kk + 1], axis=-1)
    qa, ka = O.pool_blocks(qf), O.pool_blocks(kf)
    bound = (np.linalg.norm(qa, axis=-1)[..., None]
             * np.linalg.norm(ka, axis=-1).max(axis=-1)[..., None, None])
    near = np.abs(sc - kth) <= TIE_REL * bound
    bad = mism & ~near
    assert not bad.any(), f"{int(bad.sum())} mismatches outside the near-tie window"
    assert mism.sum() <= MAX_MISMATCH_FRAC * mism.size
    return int(mism.sum())


def run_workload(nabla, w, ratios, seed=0):
    data = W.generate(w, seed)
    q, k = (nabla.from_storage(data[n], DEV) for n in "qk")
    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    for ratio in ratios:
        nb, inds = gpu_topk(nabla, q, k, ratio)
        n = check_topk(qf, kf, nb, inds, ratio)
        print("TOPK", w.name, ratio, "mismatches", n)


@pytest.mark.parametrize("name,ratios", [("tiny_f32", (0.3, 0.5)),
                                         ("small_bf16", (0.1, 0.25, 0.5, 0.9)),
                                         ("480p_bf16", (0.1, 0.3)),
                                         ("720p_bf16", (0.1,))])
def test_topk_configs(nabla, name, ratios):
    run_workload(nabla, W.WORKLOADS[name], ratios)


@pytest.mark.parametrize("B,h,D,s1,ratio", [(2, 3, 128, 37, 0.2), (1, 2, 64, 300, 0.15),
                                            (1, 2, 128, 1500, 0.05), (1, 2, 128, 1601, 0.12),
                                            (1, 2, 128, 2048, 0.02)])
def test_topk_ragged_and_large_block_counts(nabla, B, h, D, s1, ratio):
    w = W.custom(f"topk{s1}", B, h, D, 64 * s1, (s1, 1, 1), sigma=0.75, rho=0.8)
    run_workload(nabla, w, (ratio,), seed=5)


@pytest.mark.parametrize("ratio,expect", [(0.0, 0), (0.01, 0), (1.0 / 16, 1), (1.0, 16),
                                          (7.5, 16)])
def test_topk_count_edges(nabla, ratio, expect):
    """topk = min(s1, floor(ratio * s1)) at s1 = 16: zero keeps nothing, one keeps
    each row's argmax, s1 and more keep every block."""
    w = W.WORKLOADS["tiny_f32"]
    data = W.generate(w, 1)
    q, k = (nabla.from_storage(data[n], DEV) for n in "qk")
    nb, inds = gpu_topk(nabla, q, k, ratio)
    assert np.all(nb == expect)
    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    check_topk(qf, kf, nb, inds, ratio)
    if expect == w.s1:
        assert np.array_equal(inds, np.broadcast_to(np.arange(w.s1), inds.shape))
    if expect == 1:
        sc = O.topk_scores(qf, kf)
        assert np.array_equal(inds[..., 0], np.argmax(sc, axis=-1))


def _block_constant(means):
    """[1, S, h, D] f32 whose every token equals its block's mean; means is [h, s1, D]."""
    h, s1, D = means.shape
    x = np.repeat(means.transpose(1, 0, 2)[:, None], 64, axis=1)
    return np.ascontiguousarray(x.reshape(1, s1 * 64, h, D), dtype=np.float32)


def _designed(nabla, a, b, ratio, D=64, smooth=True):
    """Scores a_i * b[head, j] (exact in float32): the GPU must equal the oracle
    exactly, ties (equal b) resolved toward the higher block index.  smooth=False
    compares with a stable sort of the exact products instead (for scores whose
    fp64 smooth-k subtraction would itself round)."""
    h, s1 = b.shape
    qm = np.zeros((h, s1, D), np.float32)
    qm[:, :, 0] = a[None, :]
    km = np.zeros((h, s1, D), np.float32)
    km[:, :, 0] = b
    q, k = _block_constant(qm), _block_constant(km)
    nb, inds = gpu_topk(nabla, torch.from_numpy(q).to(DEV), torch.from_numpy(k).to(DEV), ratio)
    got = to_mask(nb, inds, s1)
    if not smooth:
        kk = O.topk_count(s1, ratio)
        prod = a.astype(np.float64)[None, :, None] * b.astype(np.float64)[:, None, :]
        order = np.argsort(prod, axis=-1, kind="stable")[None]
        want = np.zeros(got.shape, dtype=bool)
        np.put_along_axis(want, order[..., s1 - kk:], True, axis=-1)
        assert np.all(nb == kk)
        assert np.array_equal(got, want)
        return got
    ref = O.topk_mask(q.astype(np.float64), k.astype(np.float64), ratio)
    assert np.array_equal(nb, ref["kv_nb"])
    assert np.array_equal(got, ref["mask"])
    return got


@pytest.mark.parametrize("s1", [200, 1024])
@pytest.mark.parametrize("ratio", [0.1, 0.5])
def test_topk_exact_ties_and_signs(nabla, s1, ratio):
    """Nine integer levels in [-4, 4], both signs of row scale, and all-tie rows
    (a_i = 0): the cut runs through runs of equal scores."""
    rng = np.random.default_rng(21)
    a = np.array([0.0, 1.0, -1.0, 0.5], np.float32)[np.arange(s1) % 4]
    b = rng.integers(-4, 5, size=(2, s1)).astype(np.float32)
    got = _designed(nabla, a, b, ratio)
    kk = O.topk_count(s1, ratio)
    for i in range(0, s1, 4):  # a_i = 0: every score ties, the last kk blocks stay
        assert np.array_equal(np.nonzero(got[0, 0, i])[0], np.arange(s1 - kk, s1))


@pytest.mark.parametrize("s1", [256, 1536])
def test_topk_wide_key_range(nabla, s1):
    """Scores +-2^e for e in [-60, 60]: the keys span nearly all 2^32 patterns,
    so the selector narrows the range before the per-lane lists."""
    rng = np.random.default_rng(22)
    e = rng.integers(-60, 61, size=(2, s1))
    sgn = np.where(rng.random((2, s1)) < 0.5, -1.0, 1.0)
    b = (sgn * np.exp2(e.astype(np.float64))).astype(np.float32)
    b[:, : s1 // 8] = b[:, s1 // 8: s1 // 4]  # duplicated blocks: ties across the range
    a = np.array([1.0, -1.0, 0.25, 0.0], np.float32)[np.arange(s1) % 4]
    _designed(nabla, a, b, 0.3, smooth=False)


def test_topk_reuses_workspace_and_side_stream(nabla):
    """Caller-supplied workspace and outputs on a non-default stream give the
    same result as the allocating call."""
    w = W.WORKLOADS["small_bf16"]
    data = W.generate(w, 2)
    q, k = (nabla.from_storage(data[n], DEV) for n in "qk")
    nb0, inds0 = nabla.nabla_build_mask_topk(q, k, 0.2)
    ws = torch.empty(nabla.nabla_build_mask_workspace_bytes(w.B, w.S, w.h, w.D),
                     dtype=torch.uint8, device=DEV)
    nb = torch.full_like(nb0, -7)
    inds = torch.full_like(inds0, -7)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nabla.nabla_build_mask_topk(q, k, 0.2, nb, inds, ws, stream=s)
    s.synchronize()
    assert torch.equal(nb, nb0)
    kk = int(nb0[0, 0, 0])
    assert torch.equal(inds[..., :kk], inds0[..., :kk])
