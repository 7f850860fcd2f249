"""The multi-rank host path on CPU: two gloo ranks shard the rows of one
batch, each scans its block (here with the oracle: no GPU), and the gathered
result equals the single-process result; the step-time reduction is the max
over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from linear_recurrence_scan_gb300.sharding import max_over_ranks, shard_rows


def test_shard_rows_partition():
    for n in (0, 1, 7, 8, 4096, 4097):
        for w in (1, 2, 3, 8):
            blocks = [shard_rows(n, r, w) for r in range(w)]
            assert blocks[0][0] == 0 and blocks[-1][1] == n
            for (a, b), (c, d) in zip(blocks, blocks[1:]):
                assert b == c
            sizes = [b - a for a, b in blocks]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_rows(8, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from linear_recurrence_scan_gb300 import synthetic
        b = synthetic.workload_batch("gae_returns_4096x1024", N=37, T=64)
        s, e = shard_rows(37, rank, world)
        part = oracle.gae(b["rewards"][s:e], b["values"][s:e], b["terminateds"][s:e], None,
                          0.99, 0.95, None, b["last_value"][s:e])
        gathered = [None] * world
        dist.all_gather_object(gathered, (s, part))
        slow = max_over_ranks(float(rank + 1) * 10.0)
        if rank == 0:
            q.put((gathered, slow))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_without_exchange():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, slow = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    from linear_recurrence_scan_gb300 import synthetic
    b = synthetic.workload_batch("gae_returns_4096x1024", N=37, T=64)
    full = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, 0.99, 0.95, None,
                      b["last_value"])
    stitched = np.concatenate([p for _, p in sorted(gathered, key=lambda x: x[0])])
    np.testing.assert_array_equal(stitched, full)
    assert slow == 20.0
