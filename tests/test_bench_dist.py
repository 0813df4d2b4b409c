"""The bench's multi-rank aggregation on CPU: two gloo ranks on 127.0.0.1.
Each rank times its own replica; the job's time is the slowest rank's, per
timing, and the job's throughput counts every rank's units over that time.
The reference arm runs on rank 0 only; the other ranks exit without work."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # rank r reports (10 + r, 100 - r) ms: the max is (10 + ws - 1, 100)
        got = bench.max_over_ranks([10.0 + rank, 100.0 - rank], ws, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ws, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(ws):
        assert results[r] == [11.0, 100.0], (r, results[r])


def test_max_over_ranks_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]


def test_job_throughput_counts_every_rank():
    import bench
    # 2 ranks x 5e12 flops/step x 10 steps over the slowest rank's 100 ms
    assert bench.job_throughput(2, 5e12, 10, 100.0) == pytest.approx(1e15)
    assert bench.job_throughput(1, 5e12, 10, 100.0) == pytest.approx(5e14)


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
