"""Multi-rank host logic on CPU (world size 2, gloo).

The indexer shards by request / query / token with no data-path exchange; the
one exchange a chunk-range split of a single request would need is a merge of
per-shard top-k lists.  These tests check, with real gloo ranks:
  - merging each rank's top-k (score, id) lists and re-selecting gives the
    global top-k (ties to the lower id survive the merge);
  - the benchmark's max-over-ranks timing reduction.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fn, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    except Exception as e:  # surface failures to the parent
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    return out


def _shard_merge(rank, world):
    import oracle
    orc = oracle.get()
    rng = np.random.default_rng(7)
    n, k = 5000, 512
    x = rng.integers(-20, 20, n).astype(np.float64)  # heavy ties across shards
    ids = np.arange(n)
    lo, hi = rank * n // world, (rank + 1) * n // world
    idx, sc, m = orc.topk(ids[lo:hi], x[lo:hi], k)
    local = torch.tensor(np.stack([idx.astype(np.float64), sc]), dtype=torch.float64)
    gathered = [torch.zeros_like(local) for _ in range(world)]
    dist.all_gather(gathered, local)
    cand_ids, cand_x = [], []
    for g in gathered:
        sel = g[0].numpy() >= 0
        cand_ids.append(g[0].numpy()[sel].astype(np.int64))
        cand_x.append(g[1].numpy()[sel])
    merged, _, _ = orc.topk(np.concatenate(cand_ids), np.concatenate(cand_x), k)
    want, _, _ = orc.topk(ids, x, k)
    return bool((merged == want).all())


def _max_time(rank, world):
    sys.path.insert(0, ROOT)
    import bench
    return bench.reduce_max(10.0 + rank, torch.device("cpu"), world)


def test_shard_topk_merge_equals_global_topk():
    out = _run(_shard_merge)
    assert out == {0: True, 1: True}, out


def test_max_over_ranks_timing():
    out = _run(_max_time)
    assert out == {0: 11.0, 1: 11.0}, out
