"""The multi-GPU form of the benchmark: replicas only (the GEMM has no
exchange step), so N ranks each run the whole workload and the job's step
time is the slowest rank's.  Checked here with two gloo ranks on CPU: every
rank gets the maximum, the whole-job value counts every rank's work, and
the reference arm's non-zero ranks leave without work."""
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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    # rank r: timed region (3 + r) ms over 3 steps; launches 0.5 + r ms each
    totals = bench.job_step_ms(3.0 * (1 + rank), [0.5 + rank] * 3, 3, False, world)
    flushed = bench.job_step_ms(3.0 * (1 + rank), [0.5 + rank] * 3, 3, True, world)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, totals, flushed))


def test_two_ranks_take_the_slowest_step():
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
    # step times 1 and 2 ms (timed region) or 0.5 and 1.5 ms (per launch): both ranks see the max
    assert [r[1] for r in res] == [2.0, 2.0]
    assert [r[2] for r in res] == [1.5, 1.5]


def test_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 1e12 FLOP per rank per step, 2 ranks, slowest step 1 ms: 2e15 FLOP/s = 2000 TFLOP/s
    assert bench.job_value(1e12, 2, 1.0) == pytest.approx(2000.0)
    assert bench.job_value(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
