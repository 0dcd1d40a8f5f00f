"""bench.py's multi-rank host logic on CPU: two gloo ranks (no GPU needed).

The GPU arm runs one replica per rank and reports the max over ranks of the
timed region; the reference arm (the CPU oracle) runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        results[rank] = {
            "max": bench.reduce_max(1.5 + rank, world, "cpu"),
            "ref": bench.run_reference(type("A", (), {"workload": "pr1", "steps": 1, "warmup": 0})(), rank, world)
            if rank != 0 else "skipped",
        }
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_only_rank0_reports():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        mp.start_processes(_worker, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        res = dict(results)
    assert res[0]["max"] == 2.5 and res[1]["max"] == 2.5
    assert res[1]["ref"] is None  # non-zero ranks print nothing and do no oracle work
