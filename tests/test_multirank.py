"""The bench's multi-rank aggregation with two gloo ranks on CPU: each rank
decodes its own batch (replicas), the job rate is all ranks' beam-steps over
the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units = 1000.0 * (rank + 1)          # uneven work per rank
    ms = 10.0 if rank == 0 else 40.0     # rank 1 is the slowest
    rate, max_ms = bench.job_rate(units, ms, dist)
    # the graph timing runs on every rank or on none: rank 1's failed
    # capture makes both fall back
    both = bench.all_ranks_agree(True, dist)
    one_failed = bench.all_ranks_agree(rank != 1, dist)
    out[rank] = (rate, max_ms, both, one_failed)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        rate, max_ms, both, one_failed = out[r]
        assert max_ms == 40.0
        assert rate == pytest.approx(3000.0 / 0.040)
        assert both is True and one_failed is False


def test_single_process_rate():
    import bench
    rate, ms = bench.job_rate(98304.0, 6.5)
    assert rate == pytest.approx(98304 / 0.0065)
    assert bench.all_ranks_agree(True) and not bench.all_ranks_agree(False)
