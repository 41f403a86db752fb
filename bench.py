#!/usr/bin/env python3
"""Benchmark of the NABLA hot path on GB300: mask build + block-sparse attention.

One step = nabla_build_mask (pool -> pooled map -> select/CSR) followed by
nabla_attn_fwd over the kept 64x64 blocks, on one batch of the seeded synthetic
workload (default: the 720p-like latent, B=1, h=24, D=128, S=98,304, thr=0.9,
STA half-widths (3,1,1)).  Prints ONE JSON line (rank 0).

  value       kept-block attention TFLOP/s over the whole step (mask build
              included), inputs resident in HBM, CUDA-event timed;
  e2e         the same metric with q/k/v copied from pinned host memory and o
              copied back inside the timed region, every step (the copies are
              double-buffered on two copy streams and overlap the compute);
  roofline    the dominant kernel (attention) against the measured bf16 peak;
              mask_roofline: the mask builder against measured HBM bandwidth;
  cpu_baseline the fp64 oracle on a bounded sample, timed on the host cores.
`--impl reference` times the oracle itself (the reference arm of this repo).
Multi-GPU (torchrun): independent replicas, one per GPU, max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_attention_nablat_gb300 import workloads as W  # noqa: E402

METRIC = "NABLA attn fwd TFLOP/s on kept blocks (+dense-equiv); mask-build HBM GB/s"
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# launch-list capture of the workload, with the kernel versions the capture saw; an
# entry is dropped (reported as null) when its kernels change.  Workloads not
# captured: null.
NCU_TRAFFIC = {
    "720p_bf16": {
        "attention": {"bytes": 12.9557e9,
                      "source": "ncu launch list, 720p, attn_tc_kernel with the "
                                "entry-count-phased walk order"},
        "mask": {"bytes": 1.8263e9,
                 "source": "ncu launch list, 720p, pool + pooled_map + select kernels"},
    }
}
# the library kernels one step launches: pool, pooled map, select, attention
KERNELS_PER_STEP = 4
MASK_KERNELS = "mask build (pool + map + select)"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def traffic_bytes(w, part):
    e = NCU_TRAFFIC.get(w.name, {}).get(part)
    return None if e is None else e["bytes"]


def traffic_source(w, part):
    e = NCU_TRAFFIC.get(w.name, {}).get(part)
    return None if e is None else e["source"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def mask_bytes(w, total_kept_blocks: int) -> float:
    """Algorithmic bytes of one mask build: read q and k once, read the STA
    window once, write kv_nb and the kept kv_inds entries."""
    esz = 2 if w.dtype == "bf16" else 4
    return (2.0 * w.B * w.S * w.h * w.D * esz + w.s1 * w.s1 + 4.0 * w.B * w.h * w.s1
            + 4.0 * total_kept_blocks)


def attn_flops(w, total_kept_blocks: int) -> float:
    """QK^T and PV over each kept 64x64 block: 2 * 2 * 64 * 64 * D FLOP per block."""
    return 4.0 * 64 * 64 * w.D * total_kept_blocks


def dense_flops(w) -> float:
    return 4.0 * w.B * w.h * w.S * w.S * w.D


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id(dev) -> str:
    """nvidia-smi selector of a torch device (its UUID; nvidia-smi does not follow
    CUDA_VISIBLE_DEVICES numbering)."""
    import torch

    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if uuid is not None:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    return str(dev.index or 0)


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    return 0, 1, 0, None


def reduce_over_ranks(dist, device, total_ms: float, kept: float):
    """Replicas: the job's time is the slowest rank's timed region, its work the
    kept blocks of every rank.  Returns (max ms, summed kept blocks)."""
    if dist is None:
        return total_ms, kept
    import torch

    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    k = torch.tensor([float(kept)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(k, op=dist.ReduceOp.SUM)
    return t.item(), k.item()


def whole_job_tflops(w, kept_all: float, total_ms: float, steps: int) -> float:
    """Kept-block attention TFLOP/s of the whole job over the timed steps."""
    return attn_flops(w, kept_all) / (total_ms / steps * 1e-3) / 1e12


def oracle_sample(w, data, sta, thr, kv_nb=None, kv_inds=None, n_qblocks=8, seed=0):
    """Time the fp64 oracle on a bounded sample of the workload: the mask builder
    for one (batch, head) and the attention for n_qblocks query blocks.  Returns
    (kept FLOPs covered, seconds, description)."""
    from oracle import nabla_oracle as O

    qf = W.as_float(data["q"][:, :, :1])
    kf = W.as_float(data["k"][:, :, :1])
    t0 = time.perf_counter()
    r = O.build_mask(qf[:1], kf[:1], sta, thr)
    t_mask = time.perf_counter() - t0
    nb = r["kv_nb"] if kv_nb is None else kv_nb[:1, :1]
    inds = r["kv_inds"] if kv_inds is None else kv_inds[:1, :1]
    rng = np.random.default_rng(seed)
    qb = sorted({int(x) for x in rng.integers(0, w.s1, n_qblocks)})
    vf = W.as_float(data["v"][:1, :, :1])
    t0 = time.perf_counter()
    O.block_sparse_attention(qf[:1], kf[:1], vf, nb, inds, w.scale, [(0, 0, i) for i in qb])
    t_attn = time.perf_counter() - t0
    kept = int(sum(int(nb[0, 0, i]) for i in qb))
    desc = (f"oracle mask build for 1 of {w.B * w.h} (batch, head) pairs "
            f"({t_mask:.2f} s) + oracle attention for {len(qb)} of {w.B * w.h * w.s1} query "
            f"blocks ({t_attn:.2f} s); value = kept-block FLOPs of the sampled query "
            f"blocks / (mask time scaled to those blocks + attention time)")
    # mask time attributed pro rata to the sampled query blocks
    secs = t_attn + t_mask * len(qb) / w.s1
    return attn_flops(w, kept), secs, desc, t_mask, t_attn


def run_reference(args, w, thr):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import nabla_oracle as O

    data = W.generate(w, seed=0)
    sta = O.sta_mask(*w.grid, *w.sta_half_widths)
    n_q = 2
    for _ in range(args.warmup):
        oracle_sample(w, data, sta, thr, n_qblocks=n_q)
    flops, secs = 0.0, 0.0
    desc = ""
    for s in range(args.steps):
        f, t, desc, _, _ = oracle_sample(w, data, sta, thr, n_qblocks=n_q, seed=s + 1)
        flops += f
        secs += t
    value = flops / secs / 1e12
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "h": w.h, "D": w.D, "S": w.S, "thr": thr,
                   "sta_half_widths": list(w.sta_half_widths), "grid": list(w.grid),
                   "l2": "host run"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w, thr):
    import torch

    rank, world, local, dist = dist_setup(args.gpus)
    from block_sparse_attention_nablat_gb300 import nabla

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    nabla.load()
    data = W.generate(w, seed=rank)
    q, k, v = (nabla.from_storage(data[n], dev) for n in "qkv")
    sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=dev)
    kv_nb = torch.empty((w.B, w.h, w.s1), dtype=torch.int32, device=dev)
    kv_inds = torch.empty((w.B, w.h, w.s1, w.s1), dtype=torch.int32, device=dev)
    ws = torch.empty(nabla.nabla_build_mask_workspace_bytes(w.B, w.S, w.h, w.D),
                     dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step():
        nabla.nabla_build_mask(q, k, sta, thr, kv_nb, kv_inds, ws)
        nabla.nabla_attn_fwd(q, k, v, kv_nb, kv_inds, w.scale, o)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert nabla.nabla_get_last_device_status() == 0
    kept = int(kv_nb.sum().item())

    # timed region: K steps, events around each kernel group on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(dev)) as clocks:
        start.record(stream)
        for s in range(args.steps):
            ev[s][0].record(stream)
            nabla.nabla_build_mask(q, k, sta, thr, kv_nb, kv_inds, ws)
            ev[s][1].record(stream)
            nabla.nabla_attn_fwd(q, k, v, kv_nb, kv_inds, w.scale, o)
            ev[s][2].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    mask_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    assert nabla.nabla_get_last_device_status() == 0
    total_ms, kept_all = reduce_over_ranks(dist, dev, total_ms, kept)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(w, kept_all, total_ms, args.steps)

    # end to end through the public API: pinned host q/k/v in, o out, every step.
    # Copies run on their own streams with double-buffered device inputs and
    # outputs: the inputs of step s+1 are uploaded, and the output of step s-1
    # read back, while the attention of step s runs (after step s's mask build,
    # whose pool kernel needs all of HBM), as a prefetching input pipeline
    # would; every step still moves its inputs in and its output out inside the
    # timed region.  It runs right after the device-resident timed region and
    # before the extras below: run after the seconds-long backward extra, the
    # same loop measured 86-89 ms per step instead of 78-80.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3))
        hq.copy_(q), hk.copy_(k), hv.copy_(v)
        ho = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
        bufs = [(q, k, v, o)] + [tuple(torch.empty_like(t) for t in (q, k, v, o))]
        h2d_st, d2h_st = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        h2d_done, mask_done, d2h_done = ([ev() for _ in range(2)] for _ in range(3))

        def upload(s, after):
            b = s & 1
            with torch.cuda.stream(h2d_st):
                if after is not None:
                    h2d_st.wait_event(after)  # buffer b's previous step is done with it
                for dst, src in zip(bufs[b][:3], (hq, hk, hv)):
                    dst.copy_(src, non_blocking=True)
                h2d_done[b].record(h2d_st)

        def readback(s, after):
            b = s & 1
            with torch.cuda.stream(d2h_st):
                d2h_st.wait_event(after)  # step s's attention has finished
                ho[b].copy_(bufs[b][3], non_blocking=True)
                d2h_done[b].record(d2h_st)

        def e2e_run(steps):
            upload(0, None)
            for s in range(steps):
                b = s & 1
                dq, dk, dv, do = bufs[b]
                stream.wait_event(h2d_done[b])
                if s >= 2:
                    stream.wait_event(d2h_done[b])  # o of step s-2 has been read out
                nb2, inds2 = nabla.nabla_build_mask(dq, dk, sta, thr, kv_nb, kv_inds, ws)
                mask_done[b].record(stream)
                if s + 1 < steps:
                    upload(s + 1, mask_done[b])  # step s-1 finished before this mask build
                if s >= 1:
                    readback(s - 1, mask_done[b])
                nabla.nabla_attn_fwd(dq, dk, dv, nb2, inds2, w.scale, do)
            done = ev()
            done.record(stream)
            readback(steps - 1, done)
            stream.wait_event(d2h_done[(steps - 1) & 1])

        e2e_run(2)
        torch.cuda.synchronize()
        # host-link rates on their own (outside the timed region): the e2e figure
        # depends on them, and they differ between hosts
        tc = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        tc[0].record(h2d_st)
        upload(0, None)
        tc[1].record(h2d_st)
        tc[1].synchronize()
        tc[2].record(d2h_st)
        readback(0, tc[1])
        tc[3].record(d2h_st)
        tc[3].synchronize()
        nbytes = q.numel() * q.element_size()
        h2d_gbs = 3 * nbytes / (tc[0].elapsed_time(tc[1]) * 1e-3) / 1e9
        d2h_gbs = nbytes / (tc[2].elapsed_time(tc[3]) * 1e-3) / 1e9
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_id(dev)) as e2e_clocks:
            e0.record(stream)
            h2d_st.wait_event(e0)
            d2h_st.wait_event(e0)
            e2e_run(args.steps)
            e1.record(stream)
            torch.cuda.synchronize()
        e2e_ms = torch.tensor([e0.elapsed_time(e1) / args.steps], dtype=torch.float64,
                              device=dev)
        if dist is not None:
            dist.all_reduce(e2e_ms, op=dist.ReduceOp.MAX)
        e2e = {"value": attn_flops(w, kept_all) / (e2e_ms.item() * 1e-3) / 1e12,
               "unit": "TFLOP/s", "ms_per_step": e2e_ms.item(),
               "h2d_bytes_per_step": 3 * nbytes, "d2h_bytes_per_step": nbytes,
               "copies": "double-buffered on two copy streams, overlapping compute",
               "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "clocks": e2e_clocks.summary()}
        del bufs

    # Steps with nothing recorded between a step's mask build and its attention, as
    # a user's loop runs them (the attention's launch and prologue then overlap the
    # mask build's tail through the chained launches), against steps with an event
    # between the two, which breaks the chaining.  The two kinds alternate in pairs
    # of steps, so both run in the same thermal and power state; each pair is timed
    # by one event pair.  Not part of `value`.
    def timed_pair(split):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(2):
            nabla.nabla_build_mask(q, k, sta, thr, kv_nb, kv_inds, ws)
            if split:
                torch.cuda.Event().record(stream)
            nabla.nabla_attn_fwd(q, k, v, kv_nb, kv_inds, w.scale, o)
        b.record(stream)
        return a, b

    torch.cuda.synchronize()
    pairs = [(timed_pair(False), timed_pair(True)) for _ in range(max(1, args.steps // 4))]
    torch.cuda.synchronize()
    chained_ms = sum(c[0].elapsed_time(c[1]) for c, _ in pairs) / (2 * len(pairs))
    split_ms = sum(p[0].elapsed_time(p[1]) for _, p in pairs) / (2 * len(pairs))
    assert nabla.nabla_get_last_device_status() == 0

    # beside the step, timed on their own (not part of it): the steps either side
    # of the path, fractal flatten of a q-sized latent and its inverse, and the
    # top-k selector
    extras = None
    if not args.no_extras:
        T, Hs, Ws = w.grid[0], 8 * w.grid[1], 8 * w.grid[2]
        x6 = q.view(w.B, T, Hs, Ws, w.h, w.D)
        yf = torch.empty_like(q)
        xr = torch.empty_like(q).view(w.B, T, Hs, Ws, w.h, w.D)
        nbytes_q = q.numel() * q.element_size()
        extras = {}
        for name, fn in (("fractal_flatten", lambda: nabla.nabla_fractal_flatten(x6, 8, yf)),
                         ("fractal_unflatten",
                          lambda: nabla.nabla_fractal_unflatten(yf, T, Hs, Ws, 8, xr))):
            for _ in range(3):
                fn()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(5):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            us = a0.elapsed_time(a1) * 1e3 / 5
            gbs = 2 * nbytes_q / (us * 1e-6) / 1e9
            extras[name] = {"us": us, "gbs": gbs, "bytes": 2 * nbytes_q, "bound": "hbm",
                            "frac": gbs / load_peaks()[0]["hbm_gbs"]}
        # the top-k selector on the same q, k: pool + map +
        # top-k select; its algorithmic bytes are the mask build's without the
        # STA window
        ratio = 0.1
        nb_t = torch.empty_like(kv_nb)
        inds_t = torch.empty_like(kv_inds)
        fn = lambda: nabla.nabla_build_mask_topk(q, k, ratio, nb_t, inds_t, ws)  # noqa: E731
        for _ in range(3):
            fn()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(5):
            fn()
        a1.record(stream)
        torch.cuda.synchronize()
        us = a0.elapsed_time(a1) * 1e3 / 5
        kept_t = int(nb_t.sum().item())
        nbytes = mask_bytes(w, kept_t) - w.s1 * w.s1
        gbs = nbytes / (us * 1e-6) / 1e9
        extras["mask_topk"] = {"us": us, "topk_ratio": ratio, "kept_blocks": kept_t,
                               "gbs": gbs, "bytes": nbytes, "bound": "hbm",
                               "frac": gbs / load_peaks()[0]["hbm_gbs"]}
        assert nabla.nabla_get_last_device_status() == 0
        del yf, xr, nb_t, inds_t
        # the attention backward on the same inputs and mask, with a seeded upstream
        # gradient and the forward's log-sum-exp (nabla_attn_fwd_lse, as a training
        # step stores it); algorithmic FLOPs: the five 64x64xD products of a kept
        # block (S, dP, dV, dK, dQ); the dQ pass recomputes S and dP (seven run)
        g = nabla.from_storage(W.generate_dout(w, seed=rank), dev)
        bws = torch.empty(nabla.nabla_attn_bwd_workspace_bytes(w.B, w.S, w.h, w.D),
                          dtype=torch.uint8, device=dev)
        grads = [torch.empty_like(q) for _ in range(3)]
        o_l, lse = nabla.nabla_attn_fwd_lse(q, k, v, kv_nb, kv_inds, w.scale)
        bwd = lambda: nabla.nabla_attn_bwd(q, k, v, o_l, g, kv_nb, kv_inds, w.scale,  # noqa
                                           *grads, bws, lse=lse)
        for _ in range(2):
            bwd()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(3):
            bwd()
        a1.record(stream)
        torch.cuda.synchronize()
        bms = a0.elapsed_time(a1) / 3
        bflops = 5.0 * 2 * 64 * 64 * w.D * kept
        extras["attn_bwd"] = {"ms": bms, "tflops_kept": bflops / bms / 1e9, "bound": "tensor",
                              "frac": bflops / bms / 1e9 / load_peaks()[0][
                                  "bf16_tflops_sustained"],
                              "note": "tcgen05 for bf16, with the forward's log-sum-exp; "
                                      "frac of the sustained bf16 peak"}
        assert nabla.nabla_get_last_device_status() == 0
        del g, bws, grads, o_l, lse

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peaks, src = load_peaks()
    attn_tflops = attn_flops(w, kept) / (attn_ms * 1e-3) / 1e12
    peak_t = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    peak_b = peaks["bf16_tflops"]
    mask_gbs = mask_bytes(w, kept) / (mask_ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        from oracle import nabla_oracle as O

        nb_h, inds_h = kv_nb.cpu().numpy(), kv_inds.cpu().numpy()
        sta_h = sta.cpu().numpy()
        f, secs, desc, _, _ = oracle_sample(w, data, sta_h, thr, nb_h, inds_h,
                                            n_qblocks=args.cpu_qblocks)
        cpu = {"value": f / secs / 1e12, "unit": "TFLOP/s", "cores": host_cores(),
               "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "h": w.h, "D": w.D, "S": w.S, "thr": thr,
                   "grid": list(w.grid), "sta_half_widths": list(w.sta_half_widths),
                   "density": kept / (w.B * w.h * w.s1 * w.s1),
                   "l2": "inputs larger than L2 (q, k, v %.0f MB each), no flush" % (
                       q.numel() * q.element_size() / 1e6),
                   "parallelism": f"replicas x{world}"},
        "parts": {"mask_build_us": mask_ms * 1e3, "mask_build_gbs": mask_gbs,
                  "attn_ms": attn_ms, "attn_tflops_kept": attn_tflops,
                  "attn_tflops_dense_equiv": dense_flops(w) / (attn_ms * 1e-3) / 1e12,
                  "step_ms_chained": chained_ms, "step_ms_split": split_ms,
                  "chained_saving_us": (split_ms - chained_ms) * 1e3},
        "roofline": {"bound": "tensor", "kernel": "attention forward", "achieved": attn_tflops,
                     "peak": peak_t, "unit": "TFLOP/s", "frac": attn_tflops / peak_t,
                     "peak_source": f"{src} bf16 sustained (the kernel runs inside a long step)",
                     "peak_burst": peak_b, "frac_of_burst": attn_tflops / peak_b,
                     "traffic": traffic_bytes(w, "attention"),
                     "traffic_source": traffic_source(w, "attention")},
        "mask_roofline": {"bound": "hbm", "kernel": MASK_KERNELS, "achieved": mask_gbs,
                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": mask_gbs / peaks["hbm_gbs"], "frac_of_8000": mask_gbs / 8000.0,
                          "traffic": traffic_bytes(w, "mask"),
                          "traffic_source": traffic_source(w, "mask"),
                          "peak_source": f"{src} hbm"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "extras": extras,
        "gpu_launches": args.steps * KERNELS_PER_STEP,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


TABLE_ROWS = ([("tiny_f32", 0.9), ("small_bf16", 0.9), ("480p_bf16", 0.8), ("720p_bf16", 0.9)]
              + [("sweep_bf16", t) for t in (0.5, 0.7, 0.9, 0.99, 1.0)])


def table_cpu_leg(w, data, sta_h, thr, nb_h, inds_h, n_qblocks=8):
    """The CPU-baseline leg of one table row: the oracle as it stands, on the host
    cores -- the whole mask build (timed), its near-threshold blocks and how the GPU's
    mask compares with it, and the attention for n_qblocks query blocks of the first
    (batch, head), its time extrapolated to the whole workload by kept blocks."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import mask_tolerance as T
    from oracle import nabla_oracle as O

    qf, kf = W.as_float(data["q"]), W.as_float(data["k"])
    t0 = time.perf_counter()
    ref = O.build_mask(qf, kf, sta_h, thr)
    t_mask = time.perf_counter() - t0
    s1 = w.s1
    pos = np.arange(s1)[None, None, None, :]
    got = np.zeros(ref["mask"].shape, bool)
    sel = np.where(pos < nb_h[..., None], inds_h, s1).astype(np.int64)
    full = np.zeros(got.shape[:-1] + (s1 + 1,), bool)
    np.put_along_axis(full, sel, True, axis=-1)
    got = full[..., :s1]
    theta = T.block_margins(qf, kf, ref["p"])
    window = O.ambiguous_blocks(ref["c"], ref["t"], sta_h)
    ties = T.near_tie_blocks(ref["p"], ref["cdf_mask"], theta, sta_h)
    mism = got != ref["mask"]
    rng = np.random.default_rng(0)
    qb = sorted({int(x) for x in rng.integers(0, s1, n_qblocks)})
    vf = W.as_float(data["v"])
    t0 = time.perf_counter()
    O.block_sparse_attention(qf[:1, :, :1], kf[:1, :, :1], vf[:1, :, :1], nb_h[:1, :1],
                             inds_h[:1, :1], w.scale, [(0, 0, i) for i in qb])
    t_att = time.perf_counter() - t0
    kept_sample = int(sum(int(nb_h[0, 0, i]) for i in qb))
    total_kept = int(nb_h.sum())
    return {"kind": "oracle", "cores": host_cores(), "oracle_mask_s": t_mask,
            "oracle_attn_s_extrapolated": t_att * total_kept / max(1, kept_sample),
            "sample": f"mask: whole workload; attention: {len(qb)} query blocks of "
                      f"(b, h) = (0, 0), time scaled by kept blocks",
            "window_blocks": int(window.sum()), "near_tie_blocks": int(ties.sum()),
            "mismatches": int(mism.sum()), "mismatch_in_window": int((mism & window).sum()),
            "mismatch_near_tie_only": int((mism & ties & ~window).sum()),
            "mismatch_outside_both": int((mism & ~window & ~ties).sum()),
            "entries": int(mism.size)}


def run_table(args):
    """One JSON line per seeded configuration (and per threshold of the sweep): mask
    build and attention, each timed on its own with CUDA events, plus the oracle leg."""
    import torch
    from block_sparse_attention_nablat_gb300 import nabla

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nabla.load()
    peaks, src = load_peaks()
    stream = torch.cuda.current_stream()
    cache = {}
    rows = TABLE_ROWS if not args.table_only else [
        r for r in TABLE_ROWS if r[0] in args.table_only.split(",")]
    for name, thr in rows:
        w = W.WORKLOADS[name]
        if name not in cache:
            cache.clear()
            cache[name] = W.generate(w, seed=0)
        data = cache[name]
        q, k, v = (nabla.from_storage(data[n], dev) for n in "qkv")
        sta = nabla.nabla_sta_mask(*w.grid, *w.sta_half_widths, device=dev)
        kv_nb = torch.empty((w.B, w.h, w.s1), dtype=torch.int32, device=dev)
        kv_inds = torch.empty((w.B, w.h, w.s1, w.s1), dtype=torch.int32, device=dev)
        ws = torch.empty(nabla.nabla_build_mask_workspace_bytes(w.B, w.S, w.h, w.D),
                         dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        for _ in range(max(3, args.warmup)):
            nabla.nabla_build_mask(q, k, sta, thr, kv_nb, kv_inds, ws)
            nabla.nabla_attn_fwd(q, k, v, kv_nb, kv_inds, w.scale, o)
        torch.cuda.synchronize()
        steps = args.steps
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        with ClockSampler(gpu_id(dev)) as clocks:
            for s in range(steps):
                ev[s][0].record(stream)
                nabla.nabla_build_mask(q, k, sta, thr, kv_nb, kv_inds, ws)
                ev[s][1].record(stream)
                nabla.nabla_attn_fwd(q, k, v, kv_nb, kv_inds, w.scale, o)
                ev[s][2].record(stream)
            torch.cuda.synchronize()
        assert nabla.nabla_get_last_device_status() == 0
        mask_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
        attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
        kept = int(kv_nb.sum().item())
        mask_gbs = mask_bytes(w, kept) / (mask_ms * 1e-3) / 1e9
        kept_tf = attn_flops(w, kept) / (attn_ms * 1e-3) / 1e12
        l2 = "inputs larger than L2, no flush" if q.numel() * q.element_size() > 129e6 else \
            "inputs smaller than L2: back-to-back calls, not flushed (warm L2)"
        row = {"workload": name, "thr": thr, "dtype": w.dtype, "density": kept / (
                   w.B * w.h * w.s1 * w.s1), "kept_blocks": kept,
               "mask_us": mask_ms * 1e3, "mask_gbs": mask_gbs,
               "mask_frac_hbm": mask_gbs / peaks["hbm_gbs"],
               "attn_ms": attn_ms, "attn_tflops_kept": kept_tf,
               "attn_tflops_dense_equiv": dense_flops(w) / (attn_ms * 1e-3) / 1e12,
               "attn_frac_bf16_sustained": kept_tf / peaks["bf16_tflops_sustained"],
               "attn_frac_bf16_burst": kept_tf / peaks["bf16_tflops"],
               "attn_path": "tcgen05 bf16" if w.dtype == "bf16" else "CUDA-core fp32",
               "steps": steps, "l2": l2, "peaks": src, "clocks": clocks.summary()}
        if not args.no_cpu_baseline:
            row["cpu_baseline"] = table_cpu_leg(w, data, sta.cpu().numpy(), thr,
                                                kv_nb.cpu().numpy(), kv_inds.cpu().numpy())
        print(json.dumps(row), flush=True)
        del q, k, v, kv_nb, kv_inds, ws, o


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="720p_bf16", choices=list(W.WORKLOADS))
    ap.add_argument("--thr", type=float, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-qblocks", type=int, default=8)
    ap.add_argument("--table", action="store_true",
                    help="one line per seeded configuration and sweep threshold")
    ap.add_argument("--table-only", default="", help="comma-separated workloads of --table")
    args = ap.parse_args()
    if args.table:
        run_table(args)
        return
    w = W.WORKLOADS[args.workload]
    thr = args.thr if args.thr is not None else w.thr[0]
    if args.impl == "reference":
        run_reference(args, w, thr)
    else:
        run_ours(args, w, thr)


if __name__ == "__main__":
    main()
