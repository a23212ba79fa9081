"""Host logic of the benchmark on CPU: the multi-rank path (N independent replicas joined only
by a MAX reduction of their timings over gloo, world size 2), the whole-job throughput formula,
and the lookup of recorded DRAM traffic (valid only for its workload, schedule and source)."""
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


def test_traffic_lookup_matches_workload_schedule_and_source_hash(monkeypatch):
    import bench
    # the recorded entries apply to their own workload and schedule only
    assert bench.traffic_per_launch("attn_bwd", "llama8b_s8k", 8, 131072) is None
    assert bench.traffic_per_launch("attn_bwd", "llama8b_s128k", 16, 131072) is None
    assert bench.traffic_per_launch("no_such_kernel", "llama8b_s128k", 8, 131072) is None
    # a source change makes every figure taken on the old source unusable (null)
    monkeypatch.setattr(bench, "source_hash", lambda files: "0" * 64)
    assert bench.traffic_per_launch("attn_bwd", "llama8b_s128k", 8, 131072) is None
    assert bench.traffic_per_launch("loss_gemm", "llama8b_readout_s128k", 8192, None) is None
    # with the recorded hash each entry is found, one per workload for a shared kernel class
    monkeypatch.setattr(bench, "source_hash",
                        lambda files: next(e["sha256"] for es in bench.TRAFFIC.values()
                                           for e in (es if isinstance(es, list) else [es])
                                           if e["files"] == files))
    a = bench.traffic_per_launch("loss_gemm", "llama8b_readout_s128k", 8192, None)
    b = bench.traffic_per_launch("loss_gemm", "llama8b_mlp_s128k", 8192, None)
    assert a and b and a != b
