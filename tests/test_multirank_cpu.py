"""The replica (N > 1) timing path of bench.py on two gloo ranks on the CPU: the job time is the
slowest rank's, the job's work is every rank's, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
        value = bench.whole_job_tflops(1e12, 5, slowest, world)
        dist.barrier()
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_replica_timing_on_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree on the slowest time (20 ms) and on the whole-job value
    assert [r[1] for r in res] == [20.0, 20.0]
    expected = 2 * 1e12 * 5 / (20.0e-3) / 1e12
    assert all(r[2] == pytest.approx(expected) for r in res)


def test_reference_arm_runs_on_rank_zero_only():
    import sys
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 0

    assert bench.run_reference(A(), None, rank=1, world=2) is None
