"""The N>1 host logic of bench.py on CPU: two gloo ranks on 127.0.0.1 join the
process group through bench's own setup, meet at its barrier, agree on the
slowest rank's time, and the whole-job throughput counts both ranks' work."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(w, 10.0 + 5.0 * rank)       # rank 1 is slower
    out[rank] = slowest
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    if torch.cuda.is_available():
        pytest.skip("CPU test of the host logic (gloo)")
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_value_counts_every_rank():
    one = bench.whole_job_tflops(1, 51.54e9, 0.13)
    assert bench.whole_job_tflops(2, 51.54e9, 0.13) == pytest.approx(2 * one)
    assert one == pytest.approx(51.54e9 / 0.13e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_setup(1) == (1, 0, 0)
    assert bench.max_over_ranks(1, 3.5) == 3.5
