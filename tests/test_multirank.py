"""The N > 1 path of bench.py on CPU: two gloo ranks.

The hot path shards without any data exchange (every rank runs its own
replica of the workload), so the only cross-rank logic is the timing: the
slowest rank's time is taken (max over ranks), and the reference arm runs on
rank 0 alone while the other ranks exit without work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import argparse

    import bench
    import workloads as wl
    got = bench.reduce_max(1.5 * (rank + 1), ws)                  # each rank's total time
    dist.barrier()
    args = argparse.Namespace(warmup=3, steps=2)
    ref = bench.run_reference(args, wl.WORKLOADS["int8_pth_tiny"]) if rank != 0 else "skipped"
    out.put((rank, got, bench._dist(), ref))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_only_rank0_runs_the_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, got, d, ref = q.get(timeout=120)
        res[rank] = (got, d, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 3.0                            # max(1.5, 3.0) on both ranks
    assert res[0][1] == (2, 0, 0) and res[1][1] == (2, 1, 1)
    assert res[1][2] is None                                        # rank 1: no reference work, no line


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.5, 1) == 2.5
