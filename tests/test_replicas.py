"""The multi-GPU path runs independent replicas: the only cross-rank steps are
the timing barrier and the max-over-ranks of the step time. Checked here with
two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = 1.0 + rank * 0.5             # rank 1 is the slow replica
        got = bench.max_over_ranks(step_ms, "cpu")
        dist.barrier()
        out.put((rank, got, bench.replica_tokens_per_s(16, world, got)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tps in res:
        assert got == pytest.approx(1.5)
        assert tps == pytest.approx(2 * 16 / 1.5e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.replica_tokens_per_s(16, 1, 0.25) == pytest.approx(64000.0)
