"""The multi-rank path of bench.py on CPU: two gloo ranks.  With replicas
(one independent copy of the workload per GPU, no collective on the data
path), the only cross-rank steps are the barrier around the timed region and
the max over ranks of its duration; the reference arm runs on rank 0 alone."""
import importlib.util
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench = load_bench()
        barrier, max_over_ranks = bench.rank_tools(torch, dist, "cpu")
        barrier()
        dt = max_over_ranks(0.5 + rank)        # rank 1 is the slow one
        rate = bench.aggregate_rate(100, 4, world, dt)
        barrier()
        q.put((rank, dt, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port, world = free_port(), 2
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, dt, rate in got:
        assert dt == 1.5                       # max over ranks
        assert rate == pytest.approx(100 * 4 * world / 1.5)


def test_single_rank_tools_are_identity():
    import torch
    bench = load_bench()
    barrier, max_over_ranks = bench.rank_tools(torch, None, "cpu")
    barrier()
    assert max_over_ranks(2.5) == 2.5
    assert bench.aggregate_rate(10, 3, 1, 2.0) == 15.0


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0
    assert out.stdout.strip() == ""
