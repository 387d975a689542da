"""The N > 1 host logic of the benchmark on CPU: two gloo ranks (replicas),
a barrier, the max over ranks of the step time, and the whole-job value."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms = bench.max_over_ranks(dist, local_ms, torch.device("cpu"))
        out[rank] = (ms, bench.replica_value(1_000_000, world, ms))
        # the e2e leg runs only when every rank's host buffers fit
        out[f"agree{rank}"] = (bench.all_ranks_agree(dist, True, torch.device("cpu")),
                               bench.all_ranks_agree(dist, rank == 0, torch.device("cpu")))
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; the value counts both replicas
    assert out[0] == out[1] == (15.0, pytest.approx(2 * 1_000_000 / 0.015))
    # one rank without room turns the e2e leg off on all of them
    assert out["agree0"] == out["agree1"] == (True, False)


def test_host_fits_reads_available_memory():
    import bench
    assert bench.host_fits(0)
    assert not bench.host_fits(1 << 62)
