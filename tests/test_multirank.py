"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

The path has no exchange step (requests are independent), so N GPUs run N
replicas: each rank draws its own batch and the job's time is the slowest
rank's.  These tests check both pieces with real process groups."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from kv_cache_serving_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.dist_env()
        times = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], "cpu")
        cfg = wl.WORKLOADS["llamagen-xl"]
        w = wl.generate(cfg, seed=bench.rank_seed(cfg, r), with_kv=False)
        # every rank sees every rank's first sequence length (to compare batches)
        first = torch.tensor([float(w["seq_len"][0]), float(w["seq_len"].sum())])
        gathered = [torch.zeros(2) for _ in range(wsz)]
        dist.all_gather(gathered, first)
        out[rank] = (r, wsz, local, times, [g.tolist() for g in gathered])
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_and_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(90)
            assert p.exitcode == 0
        res = dict(out)
    for rank in range(world):
        r, wsz, local, times, gathered = res[rank]
        assert (r, wsz, local) == (rank, world, rank)
        assert times == [2.0, 10.0, 0.5]          # element-wise max over the two ranks
        assert gathered[0] != gathered[1]          # each rank drew its own batch
    assert res[0][4] == res[1][4]


def test_max_over_ranks_without_a_group_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 1.5], "cpu") == [3.0, 1.5]
