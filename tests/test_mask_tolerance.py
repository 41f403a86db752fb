"""The mask tolerance against hand-worked rows and against an emulation of the device
arithmetic (CPU only).

Sources: FastVideo API reference, page "nabla", nablaT_v2 "Map binarization" (keep when
the ascending running sum is >= 1 - thr); the stated criterion that blocks within 1e-4
of 1 - thr may differ; reading R8(b) for near ties across the cut.
"""
import math
import os

import numpy as np
import pytest

import mask_tolerance as T
from oracle import nabla_oracle as O
from block_sparse_attention_nablat_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "mask_tolerance.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line in ("window", "tie"):
                cur = {"kind": line}
                cases.append(cur)
                continue
            key, val = line.split(":", 1)
            if key in ("p", "thr", "theta"):
                vals = [float(x) for x in val.split()]
                cur[key] = np.array(vals) if key == "p" else vals[0]
            else:
                cur[key] = np.array([int(x) for x in val.split()], dtype=bool)
    return cases


CASES = _load_cases()


def test_golden_file_has_both_kinds():
    kinds = [c["kind"] for c in CASES]
    assert kinds.count("window") >= 4 and kinds.count("tie") >= 4


@pytest.mark.parametrize("case", [c for c in CASES if c["kind"] == "window"])
def test_window_golden(case):
    c = O.cdf_values(case["p"])
    got = O.ambiguous_blocks(c, O.cut_level(case["thr"]), case["sta"], 1e-4)
    assert np.array_equal(got, case["expect"]), (got, case["expect"])


@pytest.mark.parametrize("case", [c for c in CASES if c["kind"] == "tie"])
def test_near_tie_golden(case):
    got = T.near_tie_blocks(case["p"], case["keep"], case["theta"], case["sta"])
    assert np.array_equal(got, case["expect"]), (got, case["expect"])


def test_window_is_not_fooled_by_a_wrong_comparison():
    """<= instead of < and a missing STA exclusion both change window-1/window-2."""
    w1, w2 = [c for c in CASES if c["kind"] == "window"][:2]
    c = O.cdf_values(w2["p"])
    t = O.cut_level(w2["thr"])
    assert not np.array_equal(np.abs(c - t) < 1e-4, w2["expect"])  # STA not excluded
    # a window of 5e-5 half width (a mistaken tolerance) loses both flags of window-1
    c1 = O.cdf_values(w1["p"])
    assert not np.array_equal(O.ambiguous_blocks(c1, O.cut_level(w1["thr"]), None, 4e-5),
                              w1["expect"])


def test_near_tie_closed_form():
    """A dropped and a kept block closer than the summed margins are both flagged;
    well-separated rows flag nothing."""
    p = np.array([[0.1, 0.2, 0.3, 0.4], [0.1, 0.3, 0.3 * (1 + 2e-6), 0.3 - 2e-6 * 0.3]])
    keep = np.array([[False, True, True, True], [False, False, True, True]])
    got = T.near_tie_blocks(p, keep, 0.5e-5)
    assert not got[0].any()
    assert got[1, 1] and got[1, 2] and got[1, 3] and not got[1, 0]


def test_near_tie_map_shaped_inputs():
    """[B, h, s1, s1] maps with an [s1, s1] STA broadcast over the rows."""
    rng = np.random.default_rng(3)
    p = rng.random((1, 2, 4, 4))
    p /= p.sum(-1, keepdims=True)
    keep = O.cdf_keep(p, 0.7)
    sta = np.eye(4, dtype=np.uint8)
    got = T.near_tie_blocks(p, keep, 1.0, sta)  # a huge margin flags every non-STA block
    want = np.broadcast_to(~np.eye(4, dtype=bool), p.shape) & (
        keep.any(-1, keepdims=True) & (~keep).any(-1, keepdims=True))
    assert np.array_equal(got, want)


# ------------------------------------------------------------- device arithmetic
def _tf32_rna(x):
    """Round float32 to tf32 (10 explicit mantissa bits), to nearest, ties away."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = (u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)
    return u.view(np.float32)


def _to_f32(x, truncate):
    """float64 -> float32, rounded to nearest or toward zero."""
    y = x.astype(np.float32)
    if truncate:
        over = np.abs(y.astype(np.float64)) > np.abs(x)
        y = np.where(over, np.nextafter(y, np.float32(0)), y)
    return y


def _pool_cuda_cores(x, mul):
    """The CUDA-core pool: four row groups of 16 rows (rows g, g+4, ...), each summed in
    float32 in order, joined left to right, times mul.  x [B, S, h, D] float32."""
    B, S, h, D = x.shape
    xb = x.reshape(B, S // 64, 64, h, D)
    parts = []
    for g in range(4):
        acc = np.zeros((B, S // 64, h, D), np.float32)
        for r in range(16):
            acc = acc + xb[:, :, g + 4 * r]
        parts.append(acc)
    s = ((parts[0] + parts[1]) + parts[2]) + parts[3]
    return (s * np.float32(mul)).transpose(0, 2, 1, 3)


def _pool_tensor_cores(x, mul, truncate):
    """A tensor-core pool: 64 rows in four K=16 steps into an fp32 accumulator."""
    B, S, h, D = x.shape
    xb = x.reshape(B, S // 64, 64, h, D).astype(np.float64)
    acc = np.zeros((B, S // 64, h, D), np.float32)
    for st in range(4):
        acc = _to_f32(acc.astype(np.float64) + xb[:, :, 16 * st:16 * st + 16].sum(2), truncate)
    return (acc * np.float32(mul)).transpose(0, 2, 1, 3)


def _map_tf32(qm, km, truncate, cross_first=False):
    """The three-term tf32 map: 8-wide k-steps of lo*hi, hi*lo, hi*hi into an fp32
    accumulator (each step exact, then rounded or truncated to fp32)."""
    qh = _tf32_rna(qm)
    ql = _tf32_rna(qm - qh)
    kh = _tf32_rna(km)
    kl = _tf32_rna(km - kh)
    D = qm.shape[-1]
    f64 = lambda a: a.astype(np.float64)  # noqa: E731
    acc = np.zeros(qm.shape[:-1] + (km.shape[-2],), np.float32)
    terms = [(ql, kh), (qh, kl), (qh, kh)]
    order = ([(t, c) for t in range(2) for c in range(0, D, 8)] + [(2, c) for c in range(0, D, 8)]
             if cross_first else [(t, c) for c in range(0, D, 8) for t in range(3)])
    for t, c in order:
        a, b = terms[t]
        part = np.matmul(f64(a[..., c:c + 8]), np.swapaxes(f64(b[..., c:c + 8]), -1, -2))
        acc = _to_f32(f64(acc) + part, truncate)
    return acc


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "bf16"), (128, "f32")])
@pytest.mark.parametrize("pool", ["cuda_cores", "tensor_rz", "tensor_rn"])
@pytest.mark.parametrize("acc", ["rz", "rn", "rz_cross_first"])
def test_error_bound_covers_device_arithmetic(D, dtype, pool, acc):
    """The derived bound U holds for a faithful float32 / tf32 emulation of the device's
    pooling and pooled map, with truncating or rounding accumulation, on inputs drawn like
    the 720p workload (AR(1) block means, sigma 0.75) and on large-offset inputs."""
    for seed, sigma in ((0, 0.75), (1, 3.0)):
        w = W.custom("tol", 1, 2, D, 64 * 24, (6, 2, 2), sigma=sigma, rho=0.8, dtype=dtype)
        d = W.generate(w, seed)
        q, k = W.as_float(d["q"]), W.as_float(d["k"])
        s = math.log2(math.e) / math.sqrt(D)
        mul_q = np.float32(np.float32(s) * np.float32(1.0 / 64.0))
        mul_k = np.float32(1.0 / 64.0)
        if pool == "cuda_cores":
            qm, km = _pool_cuda_cores(q, mul_q), _pool_cuda_cores(k, mul_k)
        else:
            tr = pool == "tensor_rz"
            qm, km = _pool_tensor_cores(q, mul_q, tr), _pool_tensor_cores(k, mul_k, tr)
        Lt = _map_tf32(qm, km, acc.startswith("rz"), acc.endswith("cross_first"))
        L = O.pooled_logits(O.pool_blocks(q), O.pool_blocks(k)) * math.log2(math.e)
        U = T.logit_error_bound(q, k)
        err = np.abs(Lt.astype(np.float64) - L)
        assert np.all(err <= U), float((err / U).max())
        # not vacuous: the bound is within a few hundred of the emulated worst error
        assert U.max() < 500 * max(err.max(), 1e-12)


def test_block_margins_shape_and_floor():
    w = W.custom("tol", 1, 2, 64, 64 * 8, (2, 2, 2), sigma=0.5, dtype="bf16")
    d = W.generate(w, 2)
    q, k = W.as_float(d["q"]), W.as_float(d["k"])
    ref = O.build_mask(q, k, np.zeros((8, 8), np.uint8), 0.9)
    th = T.block_margins(q, k, ref["p"])
    assert th.shape == ref["p"].shape
    assert np.all(th >= T.EPS_EX2) and np.all(th < 1e-3)
