"""The N > 1 path of bench.py on the CPU: two gloo ranks (world_size 2).

Each rank runs its own replica of the workload (seed = rank); the only
cross-rank step is the max over ranks of the timed region, taken with one
all_reduce.  Nothing here touches a GPU.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.max_over_ranks(1.5 + rank, dist)
    w = bench.replica_workload(1, rank)
    first = w.q.reshape(-1)[:8].astype(np.float64)
    # the replica values differ by rank; gather the first few to compare on rank 0
    t = torch.tensor(first, dtype=torch.float64)
    got = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(got, t)
    if rank == 0:
        np.save(os.path.join(out_dir, "result.npy"),
                np.array([ms] + [g.numpy() for g in got][0].tolist()
                         + [g.numpy() for g in got][1].tolist()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_replicas(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r = np.load(tmp_path / "result.npy")
    assert r[0] == 2.5                          # max over ranks of 1.5 and 2.5
    assert not np.array_equal(r[1:9], r[9:17])  # seed = rank gives each replica its own data


def test_job_throughput_counts_every_replica():
    import bench

    # two replicas of 1 GB each in 1 ms -> 2000 GB/s for the job
    assert bench.job_throughput(1e9, 2, 1.0) == pytest.approx(2000.0)
    assert bench.max_over_ranks(3.0) == 3.0
