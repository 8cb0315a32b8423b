"""The N > 1 path of bench.py on CPU with gloo, world size 2: every rank runs
its own replica (attention needs no data exchange), the job time is the
slowest rank's, and the whole-job value counts every replica's FLOPs."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, result_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 1 is the slow replica
        mine = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]
        got = bench.max_over_ranks(mine, dist)
        result_q.put((rank, got))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1] == [15.0, 20.0]
    # 2 replicas x 1e12 FLOP x 10 steps in 15 ms -> 1333.3 TFLOP/s for the job
    assert bench.job_value(1e12, 10, 15.0, 2) == pytest.approx(2e13 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 4.0], None) == [3.0, 4.0]


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun with N > 1 the reference arm (the CPU oracle) runs and prints on
    rank 0 only; every other rank exits 0 at once, without output or work."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, cwd=root, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
