"""The benchmark's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

The decode step shards by sequence with no exchange (replicas), so the only
cross-rank operations are the ones the benchmark's timing uses: process-group
setup from the torchrun environment, a barrier around the timed region, and
the max over ranks of the measured times.  These run here with the gloo
backend; no GPU is touched.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    ws, rk, local = bench.dist_setup()
    assert (ws, rk, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"            # no CUDA in this process
    bench.barrier(ws)
    # each rank "measured" a different time; every rank must see the largest
    mx = bench.max_over_ranks(1.5 * (rank + 1), ws, "cpu")
    bench.barrier(ws)
    results[rank] = mx
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_share_the_max_time():
    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(240)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        assert dict(results) == {0: 3.0, 1: 3.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    bench.barrier(1)
