"""The oracle against its pins (CPU only).  See oracle_pins.py for the sources."""
import numpy as np
import pytest

import oracle_pins as P
from oracle import nabla_oracle as O
from block_sparse_attention_nablat_gb300 import workloads as W


def test_pool_closed_form():
    P.check_pool(O.pool_blocks)


def test_pool_vs_torch():
    P.check_pool_vs_torch(O.pool_blocks)


def test_map_closed_form():
    P.check_map(O.pooled_logits)


def test_softmax_closed_form():
    P.check_softmax(O.softmax_rows)


def test_map_softmax_vs_torch():
    P.check_map_softmax_vs_torch(O.pooled_logits, O.softmax_rows)


def test_cdf_golden_rows():
    P.check_cdf_golden(O.cdf_keep)


def test_cdf_bruteforce():
    P.check_cdf_bruteforce(O.cdf_keep)


def test_cdf_invariants():
    P.check_cdf_invariants(O.cdf_keep)


def test_cdf_thr_range():
    with pytest.raises(ValueError):
        O.cdf_keep(np.array([[0.5, 0.5]]), 0.0)
    with pytest.raises(ValueError):
        O.cdf_keep(np.array([[0.5, 0.5]]), 1.5)


def test_sta_golden():
    P.check_sta_golden(O.sta_mask)


def test_sta_counts():
    P.check_sta_counts(O.sta_mask)


def test_csr():
    P.check_csr(O.csr_from_mask)


def _tiny_inputs():
    w = W.WORKLOADS["tiny_f32"]
    d = W.generate(w)
    return w, W.as_float(d["q"]), W.as_float(d["k"]), W.as_float(d["v"])


def test_builder_vs_torch_tiny():
    w, q, k, _ = _tiny_inputs()
    sta = O.sta_mask(*w.grid, *w.sta_half_widths)
    for thr in (0.5, 0.9, 0.99, 1.0):
        P.check_builder_vs_torch(O.build_mask, q, k, sta, thr)


def test_builder_vs_torch_random_bf16_like():
    w = W.custom("t", 2, 3, 32, 1536, (2, 3, 4), sigma=0.75, rho=0.8, dtype="bf16")
    d = W.generate(w, seed=11)
    q, k = W.as_float(d["q"]), W.as_float(d["k"])
    sta = O.sta_mask(*w.grid, 1, 1, 1)
    P.check_builder_vs_torch(O.build_mask, q, k, sta, 0.8)


def test_sta_forced():
    w, q, k, _ = _tiny_inputs()
    P.check_sta_forced(O.build_mask, q, k, w.s1)


def test_builder_kept_mass():
    """Every row's kept softmax mass is at least thr (spec invariant)."""
    w, q, k, _ = _tiny_inputs()
    for thr in (0.5, 0.9):
        r = O.build_mask(q, k, np.zeros((w.s1, w.s1), np.uint8), thr)
        mass = np.where(r["mask"], r["p"], 0).sum(-1)
        assert np.all(mass >= thr - 1e-12)


def test_attention_dense():
    P.check_attention_dense(O.block_sparse_attention, O.csr_from_mask)


def test_attention_masked():
    P.check_attention_masked(O.block_sparse_attention, O.csr_from_mask)


def test_attention_closed_form():
    P.check_attention_closed_form(O.block_sparse_attention, O.csr_from_mask)


def test_attention_thr1_is_dense_tiny():
    """thr = 1 gives the full mask, and the sparse attention equals dense attention."""
    w, q, k, v = _tiny_inputs()
    r = O.build_mask(q, k, np.zeros((w.s1, w.s1), np.uint8), 1.0)
    assert r["mask"].all()
    o = O.block_sparse_attention(q, k, v, r["kv_nb"], r["kv_inds"], w.scale)
    assert np.allclose(o, P.sdpa64(q, k, v, w.scale), rtol=0, atol=1e-12)


def test_generator_deterministic_and_shaped():
    w = W.WORKLOADS["small_bf16"]
    a = W.generate(W.custom("g", 1, 2, 128, 512, (2, 2, 2), dtype="bf16"))
    b = W.generate(W.custom("g", 1, 2, 128, 512, (2, 2, 2), dtype="bf16"))
    assert all(np.array_equal(a[n], b[n]) for n in "qkv")
    assert a["q"].dtype == np.uint16 and a["q"].shape == (1, 512, 2, 128)
    assert w.s1 == 128 and w.grid[0] * w.grid[1] * w.grid[2] == w.s1
    # bf16 rounding is round-to-nearest-even
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], np.float32)
    assert np.array_equal(W.bf16_bits_to_f32(W.f32_to_bf16_bits(x)),
                          np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5], np.float32))
