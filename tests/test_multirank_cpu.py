"""The N > 1 path of bench.py on CPU with two gloo ranks: the rank environment,
the barrier, the max-over-ranks timing and the whole-job value; and the reference
arm's rule that ranks other than 0 exit without work.  The path runs independent
replicas (no data-path collective), so these host-side pieces are all it has."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    dist.barrier()
    slowest = bench.max_over_ranks(10.0 * (r + 1), torch.device("cpu"))
    value = bench.whole_job_tflops(2e12, w, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, local, slowest, value))


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(i, world, port, q)) for i in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, w, l) for r, w, l, _, _ in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, slowest, value in res:
        assert slowest == 20.0                        # the slower rank's 20 ms
        assert value == pytest.approx(2 * 2e12 / 20e-3 / 1e12)  # both ranks' work over it


def test_single_rank_max_is_the_value_itself():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""
