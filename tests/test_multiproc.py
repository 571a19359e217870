"""The multi-process (N > 1) host path of bench.py, on CPU with gloo.

The decode path has no exchange between GPUs: under torchrun every rank runs
an independent replica, the ranks meet at a barrier around the timed region,
the step time is the maximum over ranks, and rank 0 alone prints the JSON
line.  These tests run that host logic with two ranks on CPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), KIVI_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    r, w, dist = bench.dist_setup()
    assert (r, w) == (rank, ws)
    bench.barrier(dist)
    got = bench.reduce_max(1.5 + rank, dist)
    bench.barrier(dist)
    with open(os.path.join(outdir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo(tmp_path):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    vals = [float((tmp_path / f"rank{r}.txt").read_text()) for r in range(ws)]
    assert vals == [2.5, 2.5]


def test_reference_arm_two_ranks_one_line():
    """bench.py --impl reference under torchrun (2 ranks, gloo, CPU): rank 0
    times the oracle and prints one JSON line; the other rank exits 0."""
    env = dict(os.environ, KIVI_BENCH_BACKEND="gloo", KIVI_ORACLE_BUDGET_S="1", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_kivi2",
           "--gpus", "2", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us/step" and d["value"] > 0
    assert d["n_gpus"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
