"""Multi-rank (replicas) host logic of bench.py on CPU: two gloo ranks.

The hot path shards over (batch, head) with no exchange step, so N GPUs run N
independent replicas; the only cross-rank logic is the reduction of the timed
region (slowest rank) and of the work (every rank's kept blocks), and the
reference arm running on rank 0 alone.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from block_sparse_attention_nablat_gb300 import workloads as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, kept, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, k = bench.reduce_over_ranks(dist, "cpu", times[rank], kept[rank])
        out[rank] = (ms, k)
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_takes_slowest_time_and_sums_work():
    world = 2
    times, kept = [12.5, 17.25], [1000, 2400]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()  # both ranks meet on one port
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, kept, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(60)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        assert res[r] == (max(times), float(sum(kept)))


def test_single_rank_reduction_is_identity():
    assert bench.reduce_over_ranks(None, "cpu", 3.0, 7) == (3.0, 7)


def test_whole_job_value_is_total_work_over_time():
    w = W.WORKLOADS["720p_bf16"]
    kept_all, total_ms, steps = 4.0e7, 200.0, 2
    v = bench.whole_job_tflops(w, kept_all, total_ms, steps)
    assert v == pytest.approx(4 * 64 * 64 * w.D * kept_all / 0.1 / 1e12)
    # doubling the replicas (work) at the same slowest time doubles the value
    assert bench.whole_job_tflops(w, 2 * kept_all, total_ms, steps) == pytest.approx(2 * v)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 0, 2

    bench.run_reference(Args(), W.WORKLOADS["tiny_f32"], 0.9)
    assert capsys.readouterr().out == ""
