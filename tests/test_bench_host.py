"""CPU checks of bench.py's host logic: the max-over-ranks reduction on a
world_size-2 gloo group (the multi-rank path runs independent replicas and
shares only this timing reduction), the peak loader and the JSON contract of the
reference arm's helpers."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.reduce_max_over_ranks(10.0 + rank * 5.0, world)
    q.put((rank, v))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_over_ranks(3.5, 1) == 3.5


def test_peaks_fallback_or_measured():
    sys.path.insert(0, ROOT)
    import bench
    p = bench.load_peaks()
    assert p["source"] in ("measured", "fallback")
    assert p["hbm"] > 1000 and p["bf16"] > 500
