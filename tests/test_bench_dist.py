"""The multi-rank timing aggregation of bench.py over gloo, world size 2
(CPU only): time is the max over ranks, bytes the sum."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, nbytes = bench.reduce_over_ranks(10.0 + 5 * rank, 1000 * (rank + 1), True)
    q.put((rank, ms, nbytes))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0, 3000), (1, 15.0, 3000)]


def test_single_process_passthrough():
    import bench
    assert bench.reduce_over_ranks(3.5, 42, False) == (3.5, 42)


def test_step_bytes():
    import bench
    assert bench.colwise_bytes(65536, 4096, 16) == 805_568_512
    assert bench.rowwise_bytes(8192, 16640, 64) == 411_041_792
