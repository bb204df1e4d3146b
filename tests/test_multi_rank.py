"""The N > 1 host logic of bench.py, on CPU with gloo at world size 2.

One process per GPU runs its own replica of the workload (the path shards by
sequence batch with no data-path collective); the only collective is the
maximum of the ranks' step times, and rank 0 reports the whole job's rate.
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


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from paged_kv_attention_forward_gb300 import workloads as wl
    try:
        seed = bench.replica_seed(7, rank)
        b = wl.make_workload("tiny_decode", seed=seed)
        times = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 2.0 * (rank + 1)], dist, "cpu")
        acct = bench.algorithmic_bytes(b)
        rate = bench.whole_job_rate(acct["step"], world, times[0])
        dist.barrier()
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([seed, *times, rate, acct["step"], b.q.sum(dtype=np.int64)], dtype=np.float64))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_max_timing(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    assert r0[0] != r1[0]                                 # each rank its own replica seed
    assert r0[6] != r1[6]                                 # ... hence its own data
    assert r0[5] == r1[5]                                 # ... of the same shape and byte count
    assert list(r0[1:4]) == [2.0, 5.0, 4.0] == list(r1[1:4])   # element-wise max over ranks
    assert r0[4] == pytest.approx(world * r0[5] / (2.0e-3))    # whole-job rate uses the slowest rank
    assert r0[4] == r1[4]


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks([3.0, 1.0]) == [3.0, 1.0]
    assert bench.replica_seed(5, 0) == 5
    assert bench.whole_job_rate(1e9, 4, 2.0) == pytest.approx(2e12)
