"""The multi-replica timing of bench.py on CPU: two gloo ranks stand in for
two GPUs (each runs the same steps; the job's time per step is the slowest
rank's divided by the number of ranks).  The decode step itself exchanges
nothing between GPUs, so the timing reduction is the only collective."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, us, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        q.put((rank, bench.job_us_per_step(us[rank], ws, "cpu")))
    finally:
        dist.destroy_process_group()


def test_single_replica_time_is_its_own():
    assert bench.job_us_per_step(42.5, 1, "cpu") == 42.5


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    us = [10.0, 25.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, us, q))
             for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree: the slower rank's 25 us over 2 replicas
    assert got == {0: 12.5, 1: 12.5}
