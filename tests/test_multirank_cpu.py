"""Host logic of the N-replica bench on CPU ranks (gloo, world size 2): the job's
time is the slowest rank's, and the rate counts the steps of every rank."""
import multiprocessing
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.reduce_max(10.0 + 3.0 * rank, torch.device("cpu"))
    q.put((rank, m, bench.whole_job_rate(5, world, m), bench._dist()))
    dist.barrier()
    dist.destroy_process_group()


def test_bench_aggregation_over_two_gloo_ranks():
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v, d in res:
        assert m == 13.0                      # slowest rank's total
        assert abs(v - 2 * 5 / 13e-3) < 1e-9  # all ranks' steps over the slowest time
        assert d == (2, rank, 0)              # WORLD_SIZE, RANK, LOCAL_RANK from the env


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import torch

    import bench
    assert bench.reduce_max(7.5, torch.device("cpu")) == 7.5
    assert bench.whole_job_rate(10, 1, 20.0) == 500.0
