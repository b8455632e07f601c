"""The N-replica path of the benchmark (one process per GPU, no collective on
the data path): step time is the max over ranks and the rate counts every
rank's bytes. Checked with two gloo ranks on the CPU."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, gbs = bench.aggregate_ranks([2.0, 3.0][rank], 6e9, world, "cpu")
    dist.barrier()
    results[rank] = (ms, gbs)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        ms, gbs = results[r]
        assert ms == 3.0
        assert gbs == pytest.approx(2 * 6e9 / 3e-3 / 1e9)
