"""CUDA path vs the fp64 oracle, through the C ABI (needs an sm_103 GPU).

Tolerances (the pages state none; these are the bounds this repository holds its kernels to):
  mask: kv_nb / kv_inds bit-exact except (a) blocks whose oracle running sum lies within
        1e-4 of 1 - thr and that the STA does not force, and (b) blocks of a near tie
        straddling the cut whose probabilities differ by less than the summed error
        margins of the device's float32 arithmetic (derived per block in
        tests/mask_tolerance.py); mismatches must be such blocks, and at most 0.1% of
        all B*h*s1*s1 entries.  Window and near-tie mismatches are counted apart, and
        every near-tie mismatch is listed with its relative gap and margin.
  attention, given the same mask: max-abs 1e-5 (fp32), max-abs 1e-2 and
        mean-abs 1e-3 (bf16).
"""
import math
import time

import numpy as np
import pytest
import torch

import mask_tolerance as T
from block_sparse_attention_nablat_gb300 import workloads as W
from oracle import nabla_oracle as O

pytestmark = pytest.mark.gpu

AMB_TOL = 1e-4
MAX_MISMATCH_FRAC = 1e-3
TOL = {"f32": (1e-5, None), "bf16": (1e-2, 1e-3)}


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


DEV = "cuda:0"
_cache = {}


def inputs(w, seed=0):
    key = (w, seed)
    if key not in _cache:
        _cache.clear()
        d = W.generate(w, seed)
        _cache[key] = d
    return _cache[key]


def csr_to_mask(nb, inds, s1):
    """Boolean mask from the kept prefix of each CSR row; validates the prefix."""
    pos = np.arange(s1)
    valid = pos[None, None, None, :] < nb[..., None]
    sel = np.where(valid, inds, s1)
    assert np.all((sel >= 0) & (sel <= s1))
    # strictly ascending kept prefix
    d = np.diff(np.where(valid, inds, np.iinfo(np.int32).max).astype(np.int64), axis=-1)
    both = valid[..., 1:]
    assert np.all(d[both] > 0), "kv_inds prefix not strictly ascending"
    m = np.zeros(nb.shape + (s1 + 1,), dtype=bool)
    np.put_along_axis(m, sel.astype(np.int64), True, axis=-1)
    return m[..., :s1]


def check_mask(w, thr, data, nb, inds, sta):
    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    ref = O.build_mask(qf, kf, sta, thr)
    got = csr_to_mask(nb, inds, w.s1)
    assert np.array_equal(nb, got.sum(-1))
    theta = T.block_margins(qf, kf, ref["p"])
    window = O.ambiguous_blocks(ref["c"], ref["t"], sta, AMB_TOL)
    ties = T.near_tie_blocks(ref["p"], ref["cdf_mask"], theta, sta)
    amb = window | ties
    mism = got != ref["mask"]
    n_mis = int(mism.sum())
    rows, summary = T.mismatch_report(got, ref, window, ties, theta)
    for r in rows:
        print("MISMATCH", w.name, thr, r)
    bad = mism & ~amb
    assert not bad.any(), f"{int(bad.sum())} mismatches outside the admissible set: {rows[:8]}"
    assert n_mis <= MAX_MISMATCH_FRAC * mism.size
    assert np.all(got[:, :, sta.astype(bool)]), "an STA block was dropped"
    return {"density": float(got.mean()), "window": int(window.sum()),
            "near_tie": int(ties.sum()), "mismatches": n_mis,
            "mismatch_in_window": summary["in_window"],
            "mismatch_near_tie": summary["near_tie_only"],
            "strict_outside_window": summary["outside_window"],
            "worst_gap_over_margin": summary["worst_gap_over_margin"],
            "margin_median": float(np.median(theta)),
            "entries": int(mism.size), "ref": ref}


def gpu_mask(nabla, w, data, thr):
    q = nabla.from_storage(data["q"], DEV)
    k = nabla.from_storage(data["k"], DEV)
    sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=DEV)
    nb, inds = nabla.nabla_build_mask(q, k, sta, thr)
    assert nabla.nabla_get_last_device_status() == 0
    return nb.cpu().numpy(), inds.cpu().numpy(), sta.cpu().numpy()


def oracle_attention(qf, kf, vf, nb, inds, scale, qblocks=None, workers=4):
    """The oracle's block-sparse attention for the listed (b, h, i) query blocks (all if
    None), called head by head (views of that head's q, k and v), several heads at a
    time.  Returns float64 [B, S, h, D], NaN outside the listed blocks."""
    from concurrent.futures import ThreadPoolExecutor

    B, S, h, D = qf.shape
    s1 = S // 64
    if qblocks is None:
        qblocks = [(b, hh, i) for b in range(B) for hh in range(h) for i in range(s1)]
    groups = {}
    for b, hh, i in qblocks:
        groups.setdefault((b, hh), []).append(i)
    out = np.full((B, S, h, D), np.nan)

    def one(key):
        b, hh = key
        o = O.block_sparse_attention(qf[b:b + 1, :, hh:hh + 1], kf[b:b + 1, :, hh:hh + 1],
                                     vf[b:b + 1, :, hh:hh + 1], nb[b:b + 1, hh:hh + 1],
                                     inds[b:b + 1, hh:hh + 1], scale,
                                     [(0, 0, i) for i in groups[key]])
        for i in groups[key]:
            out[b, i * 64:(i + 1) * 64, hh, :] = o[0, i * 64:(i + 1) * 64, 0, :]

    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(one, sorted(groups)))
    return out


def check_attention(nabla, w, data, nb, inds, qblocks=None, seed=0):
    dev_in = [nabla.from_storage(data[n], DEV) for n in "qkv"]
    o = nabla.nabla_attn_fwd(*dev_in, torch.from_numpy(nb).to(DEV),
                             torch.from_numpy(np.ascontiguousarray(inds)).to(DEV), w.scale)
    assert nabla.nabla_get_last_device_status() == 0
    o = o.float().cpu().numpy()
    qf, kf, vf = (W.as_float(data[n]) for n in "qkv")
    ref = oracle_attention(qf, kf, vf, nb, inds, w.scale, qblocks)
    sel = ~np.isnan(ref)
    err = np.abs(o[sel] - ref[sel])
    amax, amean = TOL[w.dtype]
    assert err.max() <= amax, err.max()
    if amean is not None:
        assert err.mean() <= amean, err.mean()
    return float(err.max()), float(err.mean())


def sample_qblocks(w, n, seed=0):
    rng = np.random.default_rng(seed)
    out = set()
    while len(out) < n:
        out.add((int(rng.integers(w.B)), int(rng.integers(w.h)), int(rng.integers(w.s1))))
    # always include first and last blocks of the first head
    out |= {(0, 0, 0), (w.B - 1, w.h - 1, w.s1 - 1)}
    return sorted(out)


SMS = 152  # persistent attention CTAs: one per SM


def cover_qblocks(w, per_bh=64, seed=0):
    """Query blocks that reach every path of the attention kernel's work split.

    The kernel pairs blocks i and i + d inside each run of 2d blocks, with d = 1 or a d
    with 2d dividing s1 that it picks itself (on these grids the temporal neighbour
    d = H*W), and hands the (batch, head, pair) units round-robin to one persistent CTA
    per SM.  So for every (b, h): the first and last blocks, and random blocks together
    with their partners at d = 1, W and H*W, until at least per_bh blocks are chosen;
    and for the last (b, h), every block of the last 152 units at either stride (each
    CTA's last unit)."""
    Tg, Hg, Wg = w.grid
    strides = [d for d in (1, Wg, Hg * Wg) if 2 * d <= w.s1 and w.s1 % (2 * d) == 0]
    rng = np.random.default_rng(seed)
    out = set()
    for b in range(w.B):
        for hh in range(w.h):
            sel = {i for i in (0, 1, w.s1 - 2, w.s1 - 1) if 0 <= i < w.s1}
            while len(sel) < min(per_bh, w.s1):
                i = int(rng.integers(w.s1))
                sel.add(i)
                for d in strides:
                    sel.add(i + d if i % (2 * d) < d else i - d)
            out |= {(b, hh, i) for i in sel}
    hw = Hg * Wg
    tail = min(w.s1, 2 * hw * -(-SMS // hw), 2 * SMS + 2 * hw)
    out |= {(w.B - 1, w.h - 1, i) for i in range(w.s1 - tail, w.s1)}
    return sorted(out)


# ----------------------------------------------------------------------------- STA
@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_sta_matches_oracle(nabla, name):
    w = W.WORKLOADS[name]
    got = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=DEV).cpu().numpy()
    assert np.array_equal(got, O.sta_mask(*w.grid, *w.sta_half_widths))


@pytest.mark.parametrize("grid,half", [((1, 3, 3), (0, 1, 0)), ((3, 1, 2), (1, 0, 0)),
                                       ((5, 4, 6), (1, 2, 0)), ((32, 8, 8), (2, 1, 3))])
def test_sta_grids(nabla, grid, half):
    got = nabla.nabla_sta_mask(*grid, *half, device=DEV).cpu().numpy()
    assert np.array_equal(got, O.sta_mask(*grid, *half))


# ----------------------------------------------------------------------------- configs
SMALL = ["tiny_f32", "small_bf16"]
LARGE = ["480p_bf16", "720p_bf16", "sweep_bf16"]


@pytest.mark.parametrize("name", SMALL)
def test_small_config_full_parity(nabla, name):
    w = W.WORKLOADS[name]
    data = inputs(w)
    for thr in w.thr:
        nb, inds, sta = gpu_mask(nabla, w, data, thr)
        st = check_mask(w, thr, data, nb, inds, sta)
        err = check_attention(nabla, w, data, nb, inds)
        print("PARITY", name, thr, {k: v for k, v in st.items() if k != "ref"}, err)


@pytest.mark.parametrize("name", LARGE)
def test_large_config_parity(nabla, name):
    """Full mask parity at the configuration's size; attention on sampled query
    blocks (all 64 rows of each) with the GPU's own mask."""
    w = W.WORKLOADS[name]
    data = inputs(w)
    for n, thr in enumerate(w.thr):
        nb, inds, sta = gpu_mask(nabla, w, data, thr)
        st = check_mask(w, thr, data, nb, inds, sta)
        if thr == 1.0:
            assert np.all(nb == w.s1)
        qbs = cover_qblocks(w, 64, seed=n)
        err = check_attention(nabla, w, data, nb, inds, qbs)
        print("PARITY", name, thr, {k: v for k, v in st.items() if k != "ref"}, err,
              f"attention checked on {len(qbs)} query blocks")


@pytest.mark.slow
def test_480p_attention_every_query_block(nabla):
    """The whole 480p attention output (all 12,288 query blocks, ~8 TFLOP of fp64 on
    the host) against the oracle, with the GPU's own mask."""
    w = W.WORKLOADS["480p_bf16"]
    data = inputs(w)
    nb, inds, sta = gpu_mask(nabla, w, data, w.thr[0])
    t0 = time.perf_counter()
    err = check_attention(nabla, w, data, nb, inds)
    print("FULL480", {"max_abs": err[0], "mean_abs": err[1],
                      "kept_blocks": int(nb.sum()), "oracle_s": time.perf_counter() - t0})


def _map_from_workspace(ws, w):
    """The pooled map region of a mask-builder workspace (layout in include/nabla.h)."""
    M = -(-(w.B * w.h * w.s1 * w.D * 4) // 256) * 256
    n = w.B * w.h * w.s1 * w.s1
    return ws[4 * M:4 * M + 4 * n].view(torch.float32).reshape(w.B, w.h, w.s1, w.s1)


@pytest.mark.parametrize("name", ["tiny_f32", "small_bf16", "480p_bf16", "720p_bf16"])
def test_pooled_map_within_derived_bound(nabla, name):
    """Every entry of the device's pooled map (base-2 logits, read back from the
    workspace) lies within the error bound derived from the kernels' arithmetic
    (tests/mask_tolerance.py) of the exact fp64 logits: this pins the margins the
    near-tie allowance of the mask tolerance rests on."""
    w = W.WORKLOADS[name]
    data = inputs(w)
    q, k = (nabla.from_storage(data[n], DEV) for n in "qk")
    sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=DEV)
    ws = torch.empty(nabla.nabla_build_mask_workspace_bytes(w.B, w.S, w.h, w.D),
                     dtype=torch.uint8, device=DEV)
    nabla.nabla_build_mask(q, k, sta, w.thr[0], workspace=ws)
    assert nabla.nabla_get_last_device_status() == 0
    Ld = _map_from_workspace(ws, w).cpu().numpy().astype(np.float64)
    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    Lx = O.pooled_logits(O.pool_blocks(qf), O.pool_blocks(kf)) * math.log2(math.e)
    U = T.logit_error_bound(qf, kf)
    err = np.abs(Ld - Lx)
    ratio = err / U
    print("MAPERR", name, {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
                           "max_over_bound": float(ratio.max()),
                           "p99_over_bound": float(np.quantile(ratio, 0.99)),
                           "bound_median": float(np.median(U))})
    assert np.all(err <= U), float(ratio.max())


# ----------------------------------------------------------------------------- edge cases
def test_ragged_odd_block_count(nabla):
    w = W.custom("ragged", 2, 3, 128, 64 * 37, (37, 1, 1), sigma=0.75, rho=0.8, thr=(0.7,))
    data = inputs(w, seed=3)
    nb, inds, sta = gpu_mask(nabla, w, data, 0.7)
    check_mask(w, 0.7, data, nb, inds, sta)
    check_attention(nabla, w, data, nb, inds)


@pytest.mark.parametrize("s1,grid", [(300, (3, 10, 10)), (1500, (15, 10, 10)),
                                     (1601, (1601, 1, 1))])
def test_partial_last_column_tile(nabla, s1, grid):
    """s1 not a multiple of 128 (but of 4): the pooled map's last column tile has
    32-column pieces beyond s1, which its epilogue must skip without disturbing
    the stores still reading the staging buffers."""
    w = W.custom(f"partial{s1}", 1, 2, 128, 64 * s1, grid, sigma=0.75, rho=0.8, thr=(0.8,))
    data = inputs(w, seed=6)
    nb, inds, sta = gpu_mask(nabla, w, data, 0.8)
    check_mask(w, 0.8, data, nb, inds, sta)


def test_head_dim_64_bf16(nabla):
    w = W.custom("d64", 1, 4, 64, 64 * 24, (2, 3, 4), sigma=0.75, thr=(0.8,))
    data = inputs(w, seed=4)
    nb, inds, sta = gpu_mask(nabla, w, data, 0.8)
    check_mask(w, 0.8, data, nb, inds, sta)
    check_attention(nabla, w, data, nb, inds)


def test_head_dim_128_f32(nabla):
    w = W.custom("f32d128", 1, 2, 128, 64 * 10, (10, 1, 1), sigma=0.5, dtype="f32")
    data = inputs(w, seed=5)
    nb, inds, sta = gpu_mask(nabla, w, data, 0.9)
    check_mask(w, 0.9, data, nb, inds, sta)
    check_attention(nabla, w, data, nb, inds)


def test_single_block_sequence(nabla):
    w = W.custom("one", 1, 2, 128, 64, (1, 1, 1), dtype="bf16")
    data = inputs(w, seed=6)
    nb, inds, sta = gpu_mask(nabla, w, data, 0.9)
    assert np.all(nb == 1) and np.all(inds[..., 0] == 0)
    check_attention(nabla, w, data, nb, inds)


def test_max_blocks_2048(nabla):
    w = W.custom("max", 1, 1, 128, 64 * 2048, (32, 8, 8), sigma=0.75, rho=0.8, thr=(0.9,))
    data = inputs(w, seed=7)
    nb, inds, sta = gpu_mask(nabla, w, data, 0.9)
    check_mask(w, 0.9, data, nb, inds, sta)
    check_attention(nabla, w, data, nb, inds, sample_qblocks(w, 6))


def _block_constant(means):
    """[1, S, h, D] f32 whose every token equals its block's mean; means is [h, s1, D]."""
    h, s1, D = means.shape
    x = np.repeat(means.transpose(1, 0, 2)[:, None], 64, axis=1)
    return np.ascontiguousarray(x.reshape(1, s1 * 64, h, D), dtype=np.float32)


def _designed_rows(nabla, b, thr, D=64):
    """Pooled logits L[head, i, j] = a_i * b[head, j] / sqrt(D), with row scales
    a_i in {0, 1, 1.5, 2} (a_i = 0: a row of exact ties).  With no STA, the
    kept set is the CDF part alone; it must equal the oracle's except inside
    the 1e-4 window around 1 - thr (exact ties are resolved by index on both
    sides, so no near-tie allowance)."""
    h, s1 = b.shape
    a = np.array([0.0, 1.0, 1.5, 2.0], np.float32)[np.arange(s1) % 4]
    qm = np.zeros((h, s1, D), np.float32)
    qm[:, :, 0] = a[None, :]
    km = np.zeros((h, s1, D), np.float32)
    km[:, :, 0] = b
    q, k = _block_constant(qm), _block_constant(km)
    sta = np.zeros((s1, s1), np.uint8)
    nb, inds = nabla.nabla_build_mask(torch.from_numpy(q).to(DEV), torch.from_numpy(k).to(DEV),
                                      torch.from_numpy(sta).to(DEV), thr)
    assert nabla.nabla_get_last_device_status() == 0
    nb, inds = nb.cpu().numpy(), inds.cpu().numpy()
    ref = O.build_mask(q.astype(np.float64), k.astype(np.float64), sta, thr)
    got = csr_to_mask(nb, inds, s1)
    window = O.ambiguous_blocks(ref["c"], ref["t"], sta, AMB_TOL)
    bad = (got != ref["mask"]) & ~window
    assert not bad.any(), f"{int(bad.sum())} mismatches outside the 1e-4 window"
    assert np.array_equal(nb, got.sum(-1))
    return got


@pytest.mark.parametrize("s1", [1000, 1024])
@pytest.mark.parametrize("thr", [0.5, 0.9])
def test_select_clustered_row_overflows_first_bucket(nabla, s1, thr):
    """Most blocks sit in a 10 % band of probability while two outliers stretch
    the key range over ~90 binades: the first 32-bucket pass leaves hundreds of
    blocks in the cut bucket, more than the per-lane list holds, so the row is
    narrowed again in registers before the list and sort stages."""
    rng = np.random.default_rng(11)
    b = np.empty((2, s1), np.float32)
    for hd in range(2):
        v = 8.0 * 0.1 * rng.random(s1)           # cluster: L in [0, 0.1)
        v[-24:] = 8.0 * rng.uniform(-3.0, 0.0, 24)
        v[0], v[1] = 8.0 * 5.0, -8.0 * 60.0       # heavy and vanishing outliers
        b[hd] = rng.permutation(v)
    _designed_rows(nabla, b, thr)


@pytest.mark.parametrize("s1", [1000, 1024])
def test_select_runs_of_exact_ties(nabla, s1):
    """Four distinct logits, ~s1/4 blocks each: the cut lands inside a run of
    exact ties that the list passes narrow to a single key."""
    rng = np.random.default_rng(12)
    b = (2.0 * rng.integers(0, 4, size=(2, s1))).astype(np.float32)
    got = _designed_rows(nabla, b, 0.9)
    # rows with a_i = 0 are all ties: the kept blocks are the highest indices
    for i in range(0, s1, 4):
        kept = np.nonzero(got[0, 0, i])[0]
        assert np.array_equal(kept, np.arange(s1 - kept.size, s1))


def test_select_repeated_levels(nabla):
    """200 distinct levels, each on ~5 blocks: the final candidates hold
    exact ties, whose tie rank decides which copies of the cut level stay."""
    rng = np.random.default_rng(13)
    s1 = 1024
    b = (8.0 * 3.0 * rng.integers(0, 200, size=(2, s1)) / 200.0).astype(np.float32)
    for thr in (0.3, 0.7, 0.95):
        _designed_rows(nabla, b, thr)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_hand_made_csr_edge_rows(nabla, dtype):
    """Empty rows give zero output, single-block rows, full rows, and an
    alternating pattern; the CSR comes from the oracle, not the mask builder."""
    w = W.custom("csr", 1, 2, 64 if dtype == "f32" else 128, 64 * 9, (9, 1, 1), dtype=dtype)
    data = inputs(w, seed=8)
    s1 = w.s1
    mask = np.zeros((1, 2, s1, s1), bool)
    mask[0, 0, 1, 4] = True          # single block
    mask[0, 0, 2] = True             # full row
    mask[0, 0, 3, ::2] = True        # alternating
    mask[0, 1, 5, s1 - 1] = True     # last block only
    mask[0, 1, 6, :3] = True
    mask[0, 1, 8] = True
    # rows 0, 7 of head 0 and 0..4, 7 of head 1 are empty
    nb, inds = O.csr_from_mask(mask)
    inds = np.where(inds < 0, 0, inds).astype(np.int32)
    check_attention(nabla, w, data, nb, inds)
    o = nabla.nabla_attn_fwd(*[nabla.from_storage(data[n], DEV) for n in "qkv"],
                             torch.from_numpy(nb).to(DEV), torch.from_numpy(inds).to(DEV))
    o = o.float().cpu().numpy()
    assert np.all(o[0, 0:64, 0] == 0) and np.all(o[0, 7 * 64:8 * 64, 0] == 0)


def _jump_inputs(jumps, seed=11):
    """bf16 q, k, v (B=1, h=2, D=128, s1=8) whose logits jump along the key axis:
    every query row gets a common component 8 u (u = the first unit vector) and key
    block j of head hh gets c u for each (hh, j, c) in jumps, so that a row's scaled
    base-2 logits against block j rise by about 0.1275 * q_0 * c, q_0 = 8 + noise.
    With c = 100 every row's rise is 60 or more, past the kernel's 2^60 overflow
    test; with c = 60 only some rows pass it, and the others stay on the fast path
    with P values up to about 2^55."""
    w = W.custom("jump", 1, 2, 128, 64 * 8, (8, 1, 1))
    d = W.generate(w, seed)
    qf, kf, vf = (W.as_float(d[n]).copy() for n in "qkv")
    qf[..., 0] += 8.0
    for hh, j, c in jumps:
        kf[0, j * 64:(j + 1) * 64, hh, 0] += c
    data = {"q": W.f32_to_bf16_bits(qf), "k": W.f32_to_bf16_bits(kf),
            "v": W.f32_to_bf16_bits(vf)}
    return w, data


@pytest.mark.parametrize("jumps,partial", [
    ([(0, 5, 100.0), (1, 2, 100.0)], False),  # one jump, in the second / first entry of a step
    ([(0, 3, 100.0), (0, 6, 200.0), (1, 7, 100.0)], False),  # two jumps in a row; the last block
    ([(0, 5, 100.0), (1, 4, 100.0)], True),  # only some query blocks keep the jumping block
    ([(0, 5, 60.0), (1, 3, 60.0)], False),   # some rows rescale, the others keep big P values
], ids=["one-jump", "two-jumps", "partial-rows", "mixed-rows"])
def test_attention_rescale_path(nabla, jumps, partial):
    """A key block whose logits exceed the running maximum by 2^60 or more makes the
    kernel raise its exponent bias mid-row: O and l are rescaled through TMEM and the
    step's P is redone.  Random inputs never reach that path.  The blocks before the
    jump then carry 2^-60 or less of the weight, so an O or l left unscaled shows as an
    O(1) error; output and lse are compared with the oracle on every row."""
    w, data = _jump_inputs(jumps)
    s1 = w.s1
    mask = np.ones((1, 2, s1, s1), bool)
    if partial:
        mask[0, 0, 1::2, 5] = False   # odd query blocks of head 0 skip the jumping block
        mask[0, 1, ::3, 4] = False
    nb, inds = O.csr_from_mask(mask)
    inds = np.where(inds < 0, 0, inds).astype(np.int32)
    check_attention(nabla, w, data, nb, inds)
    qkv = [nabla.from_storage(data[n], DEV) for n in "qkv"]
    o, lse = nabla.nabla_attn_fwd_lse(*qkv, torch.from_numpy(nb).to(DEV),
                                      torch.from_numpy(inds).to(DEV), w.scale)
    assert nabla.nabla_get_last_device_status() == 0
    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    ref = O.attention_lse2(qf, kf, nb, inds, w.scale)
    got = lse.cpu().numpy().astype(np.float64)
    # lse up to about 280: fp32 ulp 3e-5, plus the logits' fp32 accumulation
    assert np.allclose(got, ref, rtol=0, atol=2e-3), float(np.abs(got - ref).max())



@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.3])
def test_attention_any_finite_scale(nabla, dtype, scale):
    """The ABI takes any finite softmax scale.  A negative scale turns the row
    maximum into a minimum of the raw scores (the kernel's sign-aware row maximum),
    zero gives a uniform softmax over the kept tokens, and a large one sharpens it;
    output and lse are compared with the oracle on every row."""
    w = W.custom("scale", 1, 2, 64 if dtype == "f32" else 128, 64 * 12, (3, 2, 2), dtype=dtype)
    data = inputs(w, seed=5)
    s1 = w.s1
    rng = np.random.default_rng(3)
    mask = rng.random((1, 2, s1, s1)) < 0.5
    mask[0, 0, 4] = False            # one empty row
    nb, inds = O.csr_from_mask(mask)
    inds = np.where(inds < 0, 0, inds).astype(np.int32)
    qkv = [nabla.from_storage(data[n], DEV) for n in "qkv"]
    o, lse = nabla.nabla_attn_fwd_lse(*qkv, torch.from_numpy(nb).to(DEV),
                                      torch.from_numpy(inds).to(DEV), scale)
    assert nabla.nabla_get_last_device_status() == 0
    qf, kf, vf = (W.as_float(data[n]) for n in "qkv")
    ref = oracle_attention(qf, kf, vf, nb, inds, scale)
    err = np.abs(o.float().cpu().numpy() - ref)
    if dtype == "f32":
        assert err.max() <= TOL["f32"][0], err.max()
    else:
        # P enters the PV product as bf16 while l sums the fp32 weights: the numerator
        # is off by at most 2^-9 sum_u p_u |v_u| / l <= 2^-9 max|v|; o is written as
        # bf16, <= 2^-9 |o|; each logit carries the fp32 accumulation error of its dot
        # product, at most delta = |scale| D 2^-24 max_su sum_i |q_si k_ui|, which
        # moves every weight by a factor within e^(+-delta) and o by <= 2 delta max|v|.
        # The fixed bounds of the other tests assume the default scale, whose flatter
        # softmax averages these errors down.
        vmax = float(np.abs(vf).max())
        dot = max(float((np.abs(qf[b, :, hh]) @ np.abs(kf[b, :, hh]).T).max())
                  for b in range(w.B) for hh in range(w.h))
        delta = abs(scale) * w.D * 2.0 ** -24 * dot
        bound = 2.0 ** -9 * (vmax + np.abs(ref)) + 2 * delta * vmax
        assert np.all(err <= bound), float((err / bound).max())
    lref = O.attention_lse2(qf, kf, nb, inds, scale)
    got = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.allclose(got[fin], lref[fin], rtol=0, atol=1e-3), float(np.abs(got[fin] - lref[fin]).max())

def test_threshold_one_is_dense(nabla):
    """thr = 1 keeps every block, and the sparse attention equals dense attention."""
    w = W.custom("dense", 1, 2, 128, 64 * 48, (3, 4, 4), sigma=0.75, rho=0.8, thr=(1.0,))
    data = inputs(w, seed=9)
    nb, inds, sta = gpu_mask(nabla, w, data, 1.0)
    assert np.all(nb == w.s1)
    o = nabla.nabla_attn_fwd(*[nabla.from_storage(data[n], DEV) for n in "qkv"],
                             torch.from_numpy(nb).to(DEV), torch.from_numpy(inds).to(DEV))
    qf, kf, vf = (torch.from_numpy(W.as_float(data[n])).double().permute(0, 2, 1, 3)
                  for n in "qkv")
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf).permute(0, 2, 1, 3)
    err = (o.double().cpu() - ref).abs()
    assert err.max().item() <= 1e-2 and err.mean().item() <= 1e-3


def test_out_of_range_index_is_reported_not_faulted(nabla):
    w = W.custom("bad", 1, 1, 128, 64 * 4, (4, 1, 1), dtype="bf16")
    data = inputs(w, seed=10)
    nb = np.full((1, 1, 4), 2, np.int32)
    inds = np.zeros((1, 1, 4, 4), np.int32)
    inds[..., 1] = 1
    inds[0, 0, 2, 1] = 4  # out of range: must be skipped and reported
    nb[0, 0, 3] = 5       # count beyond s1
    args = [nabla.from_storage(data[n], DEV) for n in "qkv"]
    nbt, indst = torch.from_numpy(nb).to(DEV), torch.from_numpy(inds).to(DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    o = nabla.nabla_attn_fwd(*args, nbt, indst)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 0.5, f"{elapsed:.2f} s: a bounded wait expired"
    assert nabla.nabla_get_last_device_status() == 5
    assert nabla.nabla_get_last_device_status() == 0  # cleared
    assert torch.isfinite(o.float()).all()


def test_mask_builder_deterministic(nabla):
    w = W.WORKLOADS["small_bf16"]
    data = inputs(w)
    a = gpu_mask(nabla, w, data, 0.9)
    b = gpu_mask(nabla, w, data, 0.9)
    assert np.array_equal(a[0], b[0])
    nb = a[0]
    for idx in np.ndindex(nb.shape):
        assert np.array_equal(a[1][idx][:nb[idx]], b[1][idx][:nb[idx]])


def _masks_equal(nb_a, inds_a, nb_b, inds_b, s1):
    a = csr_to_mask(nb_a.cpu().numpy(), inds_a.cpu().numpy(), s1)
    b = csr_to_mask(nb_b.cpu().numpy(), inds_b.cpu().numpy(), s1)
    return np.array_equal(a, b)


def test_mask_builder_on_side_stream_and_in_cuda_graph(nabla):
    """The mask build gives the same CSR when called on a non-default stream
    (ordered with the caller's other work on that stream, no extra
    synchronisation) and when captured in a CUDA graph and replayed."""
    w = W.custom("graph", 1, 16, 128, 64 * 512, (8, 8, 8), sigma=0.75, rho=0.8, thr=(0.9,))
    data = inputs(w, seed=21)
    q, k = (nabla.from_storage(data[n], DEV) for n in "qk")
    sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=DEV)
    nb0, inds0 = nabla.nabla_build_mask(q, k, sta, 0.9)
    torch.cuda.synchronize()
    check_mask(w, 0.9, data, nb0.cpu().numpy(), inds0.cpu().numpy(), sta.cpu().numpy())

    s = torch.cuda.Stream()
    kv_nb, kv_inds = torch.empty_like(nb0), torch.empty_like(inds0)
    ws = torch.empty(nabla.nabla_build_mask_workspace_bytes(w.B, w.S, w.h, w.D),
                     dtype=torch.uint8, device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kv_nb.fill_(-1)
        nabla.nabla_build_mask(q, k, sta, 0.9, kv_nb, kv_inds, ws, stream=s)
        copy_nb = kv_nb.clone()  # ordered after the join on s
    torch.cuda.synchronize()
    assert torch.equal(copy_nb, nb0)
    assert _masks_equal(kv_nb, kv_inds, nb0, inds0, w.s1)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nabla.nabla_build_mask(q, k, sta, 0.9, kv_nb, kv_inds, ws, stream=s)
    for _ in range(2):
        kv_nb.fill_(-1)
        kv_inds.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(kv_nb, nb0)
        assert _masks_equal(kv_nb, kv_inds, nb0, inds0, w.s1)
    assert nabla.nabla_get_last_device_status() == 0


def test_bounded_wait_gives_up_and_reports_timeout(nabla):
    """A device wait that nothing satisfies ends after its limit with
    NABLA_ERR_TIMEOUT recorded, and the context stays usable."""
    assert nabla.nabla_get_last_device_status() == 0
    t0 = time.perf_counter()
    nabla.nabla_selftest_bounded_wait()
    assert nabla.nabla_get_last_device_status() == 4
    assert time.perf_counter() - t0 < 5.0
    assert nabla.nabla_get_last_device_status() == 0
    x = torch.ones(1024, device=DEV)
    assert float(x.sum().item()) == 1024.0
