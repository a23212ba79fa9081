"""The benchmark's multi-rank path on CPU: N independent replicas joined only by a MAX
reduction of their timings over gloo (world size 2), and the whole-job throughput formula."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        tf, t_max = bench.job_throughput(times[rank], 5, 1e12, world, bench.torch_reduce_max("cpu"))
        out.put((rank, tf, t_max))
    finally:
        dist.destroy_process_group()


def test_job_throughput_single_rank():
    tf, t = bench.job_throughput(500.0, 5, 2e12, 1)
    assert t == 500.0
    assert tf == pytest.approx(5 * 2e12 / 0.5 / 1e12)


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    times = [400.0, 1000.0]  # rank 1 is the slow replica
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tf, t_max in res:
        assert t_max == 1000.0
        assert tf == pytest.approx(2 * 5 * 1e12 / 1.0 / 1e12)
