"""The N-GPU path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Rows (environments) are independent, so the job shards by environment with
no collective on the data path: each rank scans its own E x T shard and the
ranks only agree on the job's time (the slowest rank's).  This checks that
host logic without a GPU: the shards differ, the max-over-ranks reduction
gives every rank the slowest time, and the whole-job value counts every
rank's env-steps.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms_local = 1.5 + rank  # rank 1 is the slow one
        ms = bench._max_over_ranks(ms_local, torch.device("cpu"))
        value = bench._job_value(world, ms, steps=10)
        shard = bench._batch_cpu(rank)
        dist.barrier()
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), ms=ms, value=value,
                 rewards=shard["rewards"].numpy(), terminated=shard["terminated"].numpy())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_agree_on_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    import bench
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    # every rank sees the slowest rank's time
    assert float(r[0]["ms"]) == pytest.approx(2.5) and float(r[1]["ms"]) == pytest.approx(2.5)
    # whole-job value: both shards' env-steps for every estimator, in that time
    want = world * bench.E * bench.T * 10 / 2.5e-3  # env-steps per second per estimator
    assert float(r[0]["value"]) == pytest.approx(want) and float(r[1]["value"]) == pytest.approx(want)
    # the shards are the same shape but different environments
    assert r[0]["rewards"].shape == r[1]["rewards"].shape == (bench.E, bench.T)
    assert not np.array_equal(r[0]["rewards"], r[1]["rewards"])
    assert not np.array_equal(r[0]["terminated"], r[1]["terminated"])


def test_single_process_needs_no_group():
    import bench
    assert bench._max_over_ranks(3.25, torch.device("cpu")) == 3.25
    assert bench._job_value(1, 2.0, 4) == pytest.approx(bench.E * bench.T * 4 / 2e-3)
