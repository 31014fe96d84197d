"""bench.py's whole-job figures of an N-rank run (replicas: the slowest rank's
time, every rank's frames), exercised as two gloo ranks on the CPU, and the
reference arm's behaviour on ranks other than 0."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: device time 10 + r ms over 100 + r frames; e2e 1 + r s over 7 frames
        mx, sm = bench.job_totals([10.0 + rank, 1.0 + rank], [100 + rank, 7], "cpu")
        out.put((rank, mx, sm, bench.job_rate(sm[0], mx[0] / 1000.0), bench.job_rate(sm[1], mx[1])))
    finally:
        dist.destroy_process_group()


def test_job_totals_two_gloo_ranks():
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, mx, sm, rate, e2e_rate in results:
        assert mx == [11.0, 2.0], rank          # slowest rank's times
        assert sm == [201.0, 14.0], rank        # frames of both ranks
        assert rate == pytest.approx(201.0 / 0.011)
        assert e2e_rate == pytest.approx(14.0 / 2.0)


def test_job_totals_single_rank_unchanged():
    import bench
    assert bench.job_totals([3.5], [4], "cpu") == ([3.5], [4.0])
    assert bench.job_rate(10.0, 2.0) == 5.0
    assert bench.job_rate(10.0, 0.0) == 0.0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
