"""The benchmark's multi-rank host logic on CPU with two gloo ranks: rows are sharded (each rank
draws its own batch from its own seed, no collective on the data path), and the job is timed by
its slowest rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        total = bench.max_over_ranks(ms, w, "cpu")
        args = bench.parse(["--B", "6", "--V", "1000"])
        wl = bench.make_workload(args, "cpu", seed=r)
        # every rank sees the same job time; the shards differ
        gathered = [torch.zeros_like(wl.logits) for _ in range(w)]
        dist.all_gather(gathered, wl.logits)
        out[rank] = (total, bench.job_rows_per_s(wl.B, w, 4, total), not torch.equal(gathered[0], gathered[1]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_take_the_slowest_time():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == pytest.approx(6 * 2 * 4 / 0.015)
    assert res[0][2] and res[1][2]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_rows_per_s(1024, 1, 100, 12.0) == pytest.approx(1024 * 100 / 0.012)
