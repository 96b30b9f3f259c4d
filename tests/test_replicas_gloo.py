"""The N > 1 path of bench.py on CPU: replicas over gloo, world_size 2.

Every GPU holds the whole vocabulary, so N GPUs run N independent replicas of
the tail; the only cross-rank steps are the timing (the job's time is the
slowest rank's) and the rank-0 report.  Both are checked here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [180.0, 195.5][rank]  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        rows = bench.job_rows_per_s(8, 10, world, job_ms)
        out[rank] = (job_ms, rows)
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_replica_and_rows_add_up():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_replica, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    job_ms, rows = res[0]
    assert job_ms == 195.5
    assert rows == pytest.approx(8 * 10 * 2 / 0.1955)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_reports_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "0", "--gpus", "2"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if rank == 0:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []
