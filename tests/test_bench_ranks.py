"""The benchmark's multi-rank path on CPU (gloo, world size 2): each replica's
time is reduced with MAX, the job throughput counts every replica, and the
reference arm runs on rank 0 alone (other ranks exit 0 without work)."""
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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5 * rank, world, torch.device("cpu"))
        value = bench.job_throughput(512, 100, world, t)
        args = bench.parse_args(["--impl", "reference"])
        rc = bench.reference_arm(args, world, rank) if rank != 0 else 0
        dist.barrier()
        out.put((rank, t, value, rc))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, value, rc in res:
        assert t == 15.0                        # the slower replica's time on every rank
        assert value == pytest.approx(2 * 512 * 100 / 0.015)
        assert rc == 0
