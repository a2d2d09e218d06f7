"""The multi-rank logic of bench.py on CPU: two gloo ranks on one host.
Each rank runs an independent replica (no data-path collective); the job's
step time is the slowest rank's and its throughput counts every rank's
tokens.  The reference arm prints from rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://")
    import bench
    assert bench.dist_info() == (world, rank, rank)
    ms, value = bench.job_throughput(1.0 + rank, 1000, world, "cpu")
    out.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == pytest.approx(2.0)                  # max over ranks
        assert value == pytest.approx(2 * 1000 / 2e-3)   # both ranks' tokens


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(4.0, 500, 1) == (4.0, pytest.approx(500 / 4e-3))


def test_reference_arm_prints_from_rank_zero_only(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args(), bench.workload_by_name(bench.DEFAULT_WORKLOAD.name)) == 0
    assert capsys.readouterr().out == ""
