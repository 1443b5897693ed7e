"""The bench's N-rank path on CPU (gloo, world size 2): the ranks meet at the
barrier, the step time is the slowest rank's, the whole-job value counts
every rank's bytes, and under a multi-rank launch the reference arm runs on
rank 0 alone (the others exit at once, printing nothing)."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    import torch.multiprocessing as mp
    from tests import dist_workers
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ms = [10.0, 15.0]  # rank 1 is the slower one
    port = _free_port()
    procs = [ctx.Process(target=dist_workers.bench_rank, args=(r, 2, port, ms, q))
             for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in got:
        assert m == 15.0, (rank, m)
        assert v == pytest.approx(2 * 1e9 / 15e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, timeout=300)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    assert r.stdout.strip() == b""
