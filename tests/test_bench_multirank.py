"""The multi-rank host logic of bench.py on CPU: two gloo ranks, barrier, max over ranks,
whole-job throughput, and the reference arm printing on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    slowest = bench.reduce_max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
    value = bench.whole_job_tflops(2 * 10**12, 4, slowest, world)
    out.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == 15.0
        # 2 ranks x 4 steps x 2 TFLOP in 15 ms
        assert value == pytest.approx(2 * 4 * 2.0 / 0.015)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(10**12, 10, 1000.0, 1) == pytest.approx(10.0)  # 10 TFLOP in 1 s
