"""The N > 1 bench path on CPU with gloo ranks (world size 2): each rank runs
its own replica on its own sequence, there is no data-path collective, and
the whole-job rate is every rank's tokens over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [0.080, 0.095][rank]                   # rank 1 is the slower replica
    worst = bench._max_over_ranks(ms, world)
    rate = bench.whole_job_rate(1, worst, world)
    q.put((rank, worst, rate, bench.rank_seed(rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, rate, seed in got:
        assert worst == pytest.approx(0.095)
        assert rate == pytest.approx(2 / 0.095e-3)
        assert seed == rank                      # distinct replicas
