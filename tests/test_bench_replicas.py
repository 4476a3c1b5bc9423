"""bench.py --gpus N runs N independent replicas (one process per GPU, no collective
on the data path). The host logic that turns the per-rank timed regions into the
whole-job figure is checked here with two gloo ranks on the CPU: every rank ends with
the slowest rank's time, and microseconds per token count the tokens of all ranks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, ms_local, steps, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        out[rank] = bench.replicas_timing(ms_local[rank], steps, world, device="cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, [3.0, 5.0], 10, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(90)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        for r in range(2):
            ms, us = out[r]
            assert ms == 5.0
            assert us == pytest.approx(1e3 * 5.0 / (10 * 2))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replicas_timing(4.0, 8, 1) == (4.0, 500.0)
