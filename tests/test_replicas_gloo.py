"""The multi-GPU form of the benchmark is N independent replicas (one per
rank) with no data-path collective: only the timing is combined, as the
maximum over ranks, between barriers. These tests run that host-side logic
with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        # each rank "measured" a different time; every rank must see the max
        t = bench.max_over_ranks(10.0 + 5.0 * rank, w, torch.device("cpu"))
        bench.barrier(w)
        # every rank draws its own inputs (seed offset by rank): replicas, not copies
        cfg = dict(bench.WORKLOAD, L=64)
        h = bench.make_step_inputs(cfg, 1, None, seed_offset=1000 * r)[0]
        q.put((r, w, local, t, float(h["q"].float().sum())))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_over_ranks_and_distinct_replica_inputs():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r[:3] for r in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(r[3] == 15.0 for r in res)  # the max over ranks, on both ranks
    assert res[0][4] != res[1][4]          # each replica works on its own inputs


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)  # no-op without a process group
