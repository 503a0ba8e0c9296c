"""The N > 1 benchmark path on CPU: two gloo ranks (replicas of the layer, no
data-path collective) agree on the slowest rank's timings, and the whole-job
throughput counts every rank's tokens.  The data path itself has no
exchange, so this is the only multi-process logic there is."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r pretends its step took 1 + r ms and its end-to-end step 3 - r ms
        ms, e2e = bench.max_over_ranks([1.0 + rank, 3.0 - rank], torch.device("cpu"))
        q.put((rank, ms, e2e))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, e2e in got:
        assert ms == float(world)  # max of 1 + r
        assert e2e == 3.0          # max of 3 - r


def test_whole_job_throughput_is_weak_scaling():
    import bench
    assert bench.whole_job_throughput(1, 32, 0.5) == pytest.approx(64000.0)
    assert bench.whole_job_throughput(4, 32, 0.5) == pytest.approx(4 * 64000.0)
