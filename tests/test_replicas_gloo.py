"""The multi-rank bench path on CPU: two gloo ranks stand in for two GPUs running replicas.
The job's time is the slowest rank's, its tokens the sum over ranks (weak scaling)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    torch.distributed.barrier()
    t, n = bench.aggregate_ranks(torch, 10.0 + 5.0 * rank, 1000.0 * (rank + 1), world, "cpu")
    q.put((rank, t, n))
    torch.distributed.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_sum_the_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 15.0, 3000.0), (1, 15.0, 3000.0)]
