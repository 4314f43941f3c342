"""bench.py's multi-rank host logic with two gloo ranks on the CPU: the
barrier, the maximum over ranks (the job is as slow as its slowest
replica), the whole-job throughput of weak scaling, and the reference arm
running on rank 0 only.  One process per rank, 127.0.0.1 rendezvous."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world, device="cpu")
        t = bench.max_over_ranks(1.0 + rank, world, device="cpu")
        # each rank ran its own replica of 1e12 FLOPs; the slowest took t ms
        v = bench.job_tflops(world, 1e12, t)

        class A:  # the reference arm's arguments
            steps, warmup = 1, 0
        ref = bench.run_reference(A) if rank != 0 else "skipped"
        out.put((rank, t, v, ref))
        bench.barrier(world, device="cpu")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, t, v, ref = out.get(timeout=120)
        res[rank] = (t, v, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        t, v, ref = res[rank]
        assert t == 2.0                       # the slower rank's time, on every rank
        assert v == pytest.approx(world * 1e12 / 2e-3 / 1e12)  # 1000 TFLOP/s
    assert res[1][2] is None                  # rank 1 runs no reference work
