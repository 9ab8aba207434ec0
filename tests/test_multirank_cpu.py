"""The multi-GPU bench path's host logic on two CPU ranks (gloo, world size 2).

Sequences are independent, so ranks decode disjoint queries (weak scaling) and
only the timing scalars are reduced: the slowest rank's time and the sum of
steps and tokens.  No GPU is used here."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _load_bench()
    ids = bench.query_ids(10, rank, world, 5)
    # rank r "ran" for 10 + r ms, decoded 100 + r steps and 1000 + r tokens
    agg = bench.aggregate_ranks(dist, 10.0 + rank, 100 + rank, 1000 + rank, "cpu")
    q.put((rank, ids, agg))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_disjoint_queries_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (ids, agg)) for r, ids, agg in (q.get(timeout=120) for _ in range(2)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ids0, agg0 = res[0]
    ids1, agg1 = res[1]
    assert set(ids0).isdisjoint(ids1) and sorted(ids0 + ids1) == list(range(10))
    assert agg0 == agg1 == (11.0, 201.0, 2001.0)


def test_single_rank_aggregate_is_identity():
    bench = _load_bench()
    assert bench.aggregate_ranks(None, 5.0, 7, 9, "cpu") == (5.0, 7.0, 9.0)
    assert bench.query_ids(4, 0, 1, 6) == [0, 1, 2, 3, 0, 1]
