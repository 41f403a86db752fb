"""Host-side arithmetic of bench.py (CPU, no GPU): the algorithmic work the
roofline fractions divide by, and the clock-sample summary that decides
whether a run is kept.

The expected values are worked by hand from the definitions: attention does
QK^T and PV over each kept 64 x 64 block (2 * 2 * 64 * 64 * D FLOP); the mask
build reads q and k once, reads the STA window once and writes kv_nb and the
kept kv_inds entries.
"""
import os

import pytest

import bench
from block_sparse_attention_nablat_gb300 import workloads as W


def test_attention_flops_per_kept_block_and_dense_equivalent():
    w = W.WORKLOADS["720p_bf16"]  # B=1, h=24, D=128, S=98,304
    assert bench.attn_flops(w, 1) == 2 * 2 * 64 * 64 * 128
    assert bench.attn_flops(w, 0) == 0
    assert bench.dense_flops(w) == 4 * 24 * 98304 * 98304 * 128
    # every block kept: the kept-block count equals the dense count
    s1 = w.S // 64
    assert bench.attn_flops(w, w.B * w.h * s1 * s1) == bench.dense_flops(w)


def test_mask_bytes_720p():
    w = W.WORKLOADS["720p_bf16"]
    q_and_k = 2 * 98304 * 24 * 128 * 2  # bf16
    sta = 1536 * 1536
    kv_nb = 4 * 24 * 1536
    assert bench.mask_bytes(w, 0) == q_and_k + sta + kv_nb
    assert bench.mask_bytes(w, 10) - bench.mask_bytes(w, 0) == 40
    # the measured density of this workload (0.768) gives the 1.384 GB the
    # roofline fraction divides by
    kept = round(0.7681 * 24 * 1536 * 1536)
    assert bench.mask_bytes(w, kept) == pytest.approx(1.384e9, rel=2e-3)


def test_mask_bytes_fp32_counts_four_byte_elements():
    w = W.WORKLOADS["tiny_f32"]  # B=1, h=2, D=64, S=1024, s1=16
    assert bench.mask_bytes(w, 3) == 2 * 1024 * 2 * 64 * 4 + 16 * 16 + 4 * 2 * 16 + 4 * 3


def test_whole_job_rate():
    w = W.WORKLOADS["720p_bf16"]
    # 1e6 kept blocks in 2 steps of 10 ms each
    v = bench.whole_job_tflops(w, 1e6, 20.0, 2)
    assert v == pytest.approx(4 * 64 * 64 * 128 * 1e6 / 10e-3 / 1e12)


def _summary(rows):
    s = bench.ClockSampler("0")
    s.out.write("".join(r + "\n" for r in rows))
    return s.summary()


def test_clock_summary_median_under_load_and_reasons():
    na = "Not Active"
    rows = [
        f"0, 345, 2070, 120.0, 0x0, {na}, {na}, {na}, {na}",   # idle sample before the load
        f"0, 2070, 2070, 1100.0, 0x4, {na}, {na}, {na}, Active",
        f"0, 2010, 2070, 1390.0, 0x4, {na}, {na}, {na}, Active",
        f"0, 1995, 2070, 1400.0, 0x4, {na}, {na}, {na}, Active",
    ]
    got = _summary(rows)
    assert got["sm_mhz"] == 2010.0  # the idle sample is left out of the median
    assert got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]
    assert got["samples"] == 4


def test_clock_summary_reports_slowdowns_and_no_samples():
    na = "Not Active"
    got = _summary([f"0, 1500, 2070, 900.0, 0x8, Active, {na}, Active, {na}"])
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _summary([])["reasons"] == ["unsampled"]


def test_peaks_carry_the_keys_the_bench_reads():
    """The measured peaks file when present (written per machine, not part of
    the sources), else the fallback figures: either way the keys exist."""
    peaks, src = bench.load_peaks()
    assert src == ("measured" if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json"))
                   else "fallback")
    for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        assert float(peaks[key]) > 0
    for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        assert float(bench.PEAKS_FALLBACK[key]) > 0
