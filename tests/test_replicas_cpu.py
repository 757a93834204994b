"""The bench's multi-GPU form is independent replicas (the layer has no
exchange step on one node's data-parallel path): each rank times its own
steps and the job's rate is all ranks' tokens over the slowest rank's time.
Two gloo ranks on the CPU check that reduction."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        total_ms, value = bench.replicas_rate(times[rank], world, 4096, 10, torch.device("cpu"))
        out[rank] = (total_ms, value)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(120.0, 150.0), (150.0, 120.0)])
def test_replicas_rate_takes_the_slowest_rank(times):
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, world, port, times, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    slow = max(times)
    for r in range(world):
        total_ms, value = res[r]
        assert total_ms == slow
        assert value == pytest.approx(world * 4096 * 10 / (slow * 1e-3), rel=1e-12)


def test_replicas_rate_single_rank_is_local():
    import bench
    total_ms, value = bench.replicas_rate(200.0, 1, 4096, 10, torch.device("cpu"))
    assert total_ms == 200.0
    assert value == pytest.approx(4096 * 10 / 0.2, rel=1e-12)
