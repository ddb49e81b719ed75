"""The N > 1 bench logic on CPU: world-size-2 gloo ranks.

Each rank is an independent replica (the path shards by token, with no
collective on the data path); the job's time is the slowest rank's and its
throughput counts the calls of all ranks. The reference arm runs on rank 0
only; other ranks return without work.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.aggregate_ranks(10.0 * (rank + 1), calls_per_rank=100)
    # the reference arm prints only on rank 0
    buf = io.StringIO()
    if rank != 0:
        class A:  # never used: a non-zero rank returns before touching its arguments
            steps = warmup = None
        with redirect_stdout(buf):
            bench.run_reference(A())
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, value, buf.getvalue()))


def test_two_replicas_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, out in results:
        assert ms == pytest.approx(20.0)                 # the slowest rank's time
        assert value == pytest.approx(200 / 0.020)       # calls of both ranks / that time
        if rank != 0:
            assert out == ""
