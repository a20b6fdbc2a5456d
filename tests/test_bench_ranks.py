"""bench.py's multi-GPU host logic on the CPU: one process per rank (gloo,
world size 2), every rank gets the slowest rank's times, the whole-job value
counts every rank's bytes, and a world size that differs from --gpus is
refused before any GPU work."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    import rank_worker
    mp.spawn(rank_worker.max_over_ranks_worker, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        vals = [float(v) for v in (tmp_path / f"rank{r}.txt").read_text().split()]
        assert vals == [11.0, 20.0], (r, vals)


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks([3, 4.5], 1) == [3.0, 4.5]


def test_whole_job_value_counts_every_rank():
    import bench
    # 404,887,552 bytes per rank per step in 0.0826 ms
    one = bench.whole_job_gbs(404887552, 1, 0.0826)
    assert abs(one - 404887552 / 0.0826e-3 / 1e9) < 1e-6
    assert abs(bench.whole_job_gbs(404887552, 4, 0.0826) - 4 * one) < 1e-6


def test_gpus_must_match_world_size():
    env = dict(os.environ, WORLD_SIZE="3", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "WORLD_SIZE=3" in (r.stdout + r.stderr)
