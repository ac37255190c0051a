"""The multi-GPU path of bench.py on CPU: two gloo ranks (replicas, no data-path collective).

Each rank times its own replica; the job time is the slowest rank's (max over ranks) and the
whole-job throughput is all ranks' tokens over that time.  Under torchrun the reference arm runs
on rank 0 only; the other ranks exit without work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        my_ms = 2.0 + rank  # rank 1 is the slower replica
        ms = bench.max_over_ranks(my_ms, True, "cpu")
        out[rank] = (ms, bench.job_tokens_per_s(8192, ws, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_tokens():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, tps = res[rank]
        assert ms == 3.0
        assert tps == pytest.approx(8192 * 2 / 3.0e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload="prefill_t8192", steps=1, warmup=3, ref_tokens=1)
    bench.run_reference(args)   # returns at once: no oracle work, no output
    assert capsys.readouterr().out == ""


def test_single_rank_max_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, False, "cpu") == 1.25
    assert bench.job_tokens_per_s(32, 1, 0.5) == pytest.approx(64000.0)
