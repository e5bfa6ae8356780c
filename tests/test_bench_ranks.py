"""Host logic of the multi-GPU bench path (independent replicas), on CPU with
the gloo backend at world size 2: the job's time is the slowest rank's and the
throughput counts every rank's units."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank, 5.0 - rank, 7.0]
    got = bench.max_over_ranks(mine, device="cpu")
    q.put((rank, got, bench.job_throughput(1000, world, got[0])))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tput in res:
        assert got == [11.0, 5.0, 7.0]
        assert tput == pytest.approx(2000 / 0.011)


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]
    assert bench.job_throughput(500, 1, 250.0) == 2000.0
