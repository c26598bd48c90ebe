"""The benchmark's multi-rank path on CPU: two gloo ranks each take their
item shard; the shards partition the enlarged item set, every rank sees the
same queries, and the step time reduces to the maximum over ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from workload import CONFIGS, generate_rows, generate_side

    cfg = CONFIGS["d65k_q1k_i10k"].scaled(50, 700)
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    big, b, e = bench.item_shard(cfg, r, w)
    I = generate_rows(big, 1, b, e)
    Q = generate_side(cfg, 0)
    sig = torch.tensor([b, e, int(I.indices.astype(np.int64).sum()), int(Q.indices.astype(np.int64).sum())],
                       dtype=torch.int64)
    gathered = [torch.zeros_like(sig) for _ in range(world)]
    dist.all_gather(gathered, sig)
    t = torch.tensor([1.5 + rank])  # per-rank step time: the job time is the max
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        out.put(([g.tolist() for g in gathered], float(t.item())))
    dist.destroy_process_group()


def test_two_rank_item_shards_partition_the_item_set():
    from workload import CONFIGS, generate_rows

    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg = CONFIGS["d65k_q1k_i10k"].scaled(50, 700)
    big = cfg.scaled(cfg.n_q, cfg.n_i * world, name=cfg.name)
    assert [g[:2] for g in gathered] == [[0, 700], [700, 1400]]
    full = generate_rows(big, 1, 0, 1400)
    assert sum(g[2] for g in gathered) == int(full.indices.astype(np.int64).sum())
    assert gathered[0][3] == gathered[1][3]  # same queries on every rank
    assert tmax == 2.5
