"""The multi-GPU path of bench.py is replicas only: every rank runs the same
workload on its own GPU, the ranks meet at a barrier around the timed region,
the step time is the maximum over ranks, and the whole-job throughput is the
sum of the ranks' bytes over that time.  This host logic is checked here with
two gloo ranks on the CPU (no data-path collective exists to test)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    t_max = bench.allreduce_max(10.0 + rank, w)          # rank 1 is the slower one
    out[rank] = (t_max, bench.aggregate_gbs(4e9, t_max, w))
    # the reference arm: only rank 0 works, the others exit 0 at once
    if rank != 0:
        out[10 + rank] = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "gpus": world})(), w, rank)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_sum_the_bytes():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t_max, gbs = res[rank]
        assert t_max == pytest.approx(11.0)
        assert gbs == pytest.approx(world * 4e9 / 11e-3 / 1e9)
    assert res[11] == 0


def test_aggregate_is_whole_job_throughput():
    import bench
    assert bench.aggregate_gbs(58.5e9, 9.35, 1) == pytest.approx(58.5 / 9.35e-3)
    assert bench.aggregate_gbs(58.5e9, 9.35, 8) == pytest.approx(8 * 58.5 / 9.35e-3)
