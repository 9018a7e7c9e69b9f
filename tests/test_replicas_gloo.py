"""Replica bookkeeping of bench.py on CPU: two gloo ranks.

The verify pass has no exchange step at this scope, so N GPUs run N
independent replicas.  What needs checking without a GPU is the host side:
the process group, the max over ranks of the step time, the whole-job value
and that only rank 0 runs the reference arm.
"""
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


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch
    w, r, lr = bench.replica_env()
    dist = bench.init_replicas(w, "gloo")
    try:
        ms = bench.max_over_ranks(times[r], dist, torch.device("cpu"))
        q.put((r, w, lr, ms, bench.whole_job_gbs(w, 1.5e9, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.50, 0.75), (2.0, 1.0)])
def test_two_replicas_max_over_ranks(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    slow = max(times)
    for r, (rank, world, local, ms, gbs) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert ms == pytest.approx(slow)
        # both replicas stream 1.5 GB per step; the job is timed by the slower one
        assert gbs == pytest.approx(2 * 1.5e9 / (slow * 1e-3) / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_replicas(1, "gloo") is None
    assert bench.max_over_ranks(3.25, None, None) == 3.25
    assert bench.whole_job_gbs(1, 1e9, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
