"""The multi-process path of the benchmark on CPU ranks (gloo, world size 2):
one process per GPU, a barrier and max-over-ranks timing, no data-path
collective, rank 0 printing the single result line."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    import torch.distributed as td
    r, w, local = bench.dist_init("gloo")
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + r, w)  # rank 1 is the slow one
    rate = bench.whole_job_rate(10 ** 9, 4, slowest, w)
    out[rank] = (slowest, rate)
    td.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_on_gloo():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (2.0, 2 * 4.0 / 2.0)


def test_single_process_rate():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.dist_init() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(2 * 10 ** 9, 3, 2.0, 1) == 3.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    env = dict(os.environ, PYTHONPATH=str(ROOT))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           str(ROOT / "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    r = subprocess.run(cmd, cwd=str(ROOT), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == min(len(os.sched_getaffinity(0)), 48)
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
