"""Multi-rank host logic on CPU: world_size 2 over gloo (127.0.0.1)."""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from mixed_precision_paged_gb300 import sharding as sh
from mixed_precision_paged_gb300 import workloads as wl


def test_shard_sequences_partition_and_balance():
    lens = wl.high_concurrency_lens()
    pages = (lens.astype(np.int64) + 15) // 16
    for world in (1, 2, 4, 8):
        parts = [sh.shard_sequences(lens, r, world) for r in range(world)]
        allidx = np.concatenate(parts)
        assert np.array_equal(np.sort(allidx), np.arange(lens.size))        # disjoint cover
        loads = [pages[p].sum() for p in parts]
        assert max(loads) - min(loads) <= 2 * pages.max()                   # balanced by pages


def test_shard_kv_heads():
    assert list(sh.shard_kv_heads(8, 1, 4)) == [2, 3]
    with pytest.raises(ValueError):
        sh.shard_kv_heads(8, 0, 3)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = sh.max_over_ranks(10.0 + rank)
        ids = sh.agree_page_ids([5, 9, 2] if rank == 0 else [7], src=0)
        lens = wl.pages_shape_lens()
        mine = sh.shard_sequences(lens, rank, world)
        q.put((rank, t, ids.tolist(), mine.tolist()))
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, ids0, s0), (r1, t1, ids1, s1) = res
    assert t0 == t1 == 11.0
    assert ids0 == ids1 == [5, 9, 2]
    assert sorted(s0 + s1) == list(range(32)) and not set(s0) & set(s1)
