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


def _replica_worker(rank, world, port, q):
    """Each rank builds its replica's workload from its own seed and runs the
    forward's steps on it (the CPU oracle stands in for the device here:
    hash, rows, projection, gate); the ranks then compare results by an
    all-gather (a test-only collective: the benchmark's data path has none)."""
    import sys
    import numpy as np
    import torch
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle_glue as G
    from deepseek_v4_engram_hash_gb300 import configs, synth

    def replica(seed):
        cfg = configs.TINY.with_(seed=seed)
        st = G.hash_state(cfg, 1)
        wkv = [synth.wkv_rows(cfg, l, np.arange(cfg.N)) for l in range(cfg.n_layers)]
        qk = [synth.qk_weights(cfg, l) for l in range(cfg.n_layers)]
        h = synth.highway(cfg, np.arange(cfg.T))
        ids = synth.token_ids(cfg, "prefill.0", cfg.T)[None]
        out = [bench.oracle_forward(cfg, st, ids, 0, h, wkv, qk)]
        dec = synth.token_ids(cfg, "decode.0", 4)[None]
        for k in range(4):                        # decode steps carrying the look-back
            hk = synth.highway(cfg, [cfg.T + k])
            out.append(bench.oracle_forward(cfg, st, dec[:, k:k + 1], cfg.T + k, hk, wkv, qk))
        return np.concatenate(out)

    mine = torch.from_numpy(replica(bench.rank_seed(rank)))
    got = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    alone = [torch.from_numpy(replica(bench.rank_seed(r))) for r in range(world)]
    q.put((rank, all(torch.equal(got[r], alone[r]) for r in range(world)), not torch.equal(got[0], got[1])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_run_independent_replicas():
    """A replica's result depends only on its own seed: what each of two gloo
    ranks computes equals what one process computes for that replica alone,
    and the two replicas differ."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_replica_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=300) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same, differ in got:
        assert same, f"rank {rank}: a replica depends on more than its own seed"
        assert differ, "the two replicas ran the same sequence"
