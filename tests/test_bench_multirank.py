"""The multi-rank host logic of bench.py, on CPU: two gloo ranks (world_size 2).

With N GPUs the bench runs N independent replicas (no collective on the data path). What
the ranks share is host logic: each learns its rank from the launcher's environment, the
timed region is bracketed by a barrier, every rank adopts the slowest rank's time, and the
whole-job throughput counts the work of all ranks against that time. The same functions
run here over gloo that run over NCCL on GPUs; only rank 0 prints.
"""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        w, r, local = bench.dist_env()
        dist.barrier()
        # rank 1 is the slow one: both ranks must time the job by it
        slow = bench.max_over_ranks(1.0 + 2.0 * rank, w)
        value = bench.job_tflops(w, 1e12, slow)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, w, r, local, slow, value, None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, None, None, None, None, repr(e)))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=180) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    for rank, w, r, local, slow, value, err in results:
        assert err is None, err
        assert (w, r, local) == (world, rank, rank)
        assert slow == 3.0                                  # the slowest rank's milliseconds
        assert value == pytest.approx(2 * 1e12 / 3e-3 / 1e12)   # both replicas' work / slowest time
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5, 1) == 4.5
    assert bench.job_tflops(1, 2e12, 1.0) == pytest.approx(2000.0)


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    out = io.StringIO()
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 2})()
    with contextlib.redirect_stdout(out):
        bench.run_reference(args)
    assert out.getvalue() == ""
