"""The multi-rank path of bench.py on CPU: two gloo ranks agree on the maximum of their
timings (the slowest rank sets the job's time), the whole-job rate of replicas is the
per-rank rate times the ranks, and under a launcher the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=ws)
    try:
        # rank 0 is slower in the first timing, rank 1 in the second
        mine = [10.0 + 5.0 * (rank == 0), 3.0 + 4.0 * (rank == 1), 7.5]
        out[rank] = bench.max_over_ranks(mine, ws, "cpu")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_maximum():
    ws, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(ws, port, out), nprocs=ws, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == [15.0, 7.0, 7.5]


def test_whole_job_rate_of_replicas():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job(3138.0, 1) == 3138.0
    assert bench.whole_job(3138.0, 4) == 4 * 3138.0
    assert bench.max_over_ranks([1.0, 2.0], 1, "cpu") == [1.0, 2.0]


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
