"""The multi-process (replicas) path of bench.py on the CPU: gloo, world size 2.

On N GPUs every rank runs its own replica of the workload (no collective on the data
path); the job's time is the slowest rank's and its value the work of all ranks over
that time.  The reference arm runs on rank 0 alone; the other ranks exit 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    # rank 0 is the slow one on the first value, rank 1 on the second
    got = bench.reduce_max([10.0 if rank == 0 else 7.0, 1.0 if rank == 0 else 3.5], dist, "cpu")
    q.put((rank, r, w, local, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, local, got in out:
        assert (r, w, local) == (rank, 2, rank)
        assert got == [10.0, 3.5]


def test_job_value_is_the_work_of_all_ranks_over_the_slowest_time():
    import bench
    # 2 ranks x 100 steps x 1e12 FLOP in 50 s -> 4 TFLOP/s for the job
    assert bench.job_value(2, 100, 1e12, 50.0) == pytest.approx(4.0)
    assert bench.job_value(1, 100, 1e12, 50.0) == pytest.approx(2.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1", "--gpus", "2",
           "--reference-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
