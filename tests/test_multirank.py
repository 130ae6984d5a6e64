"""bench.py's multi-process host logic with world_size 2 on the CPU (gloo): rank set-up,
barrier, max-over-ranks step time and the whole-job throughput; and the reference arm's
rule that only rank 0 runs and prints.  No GPU involved."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench.dist_setup("gloo")
    bench.barrier(got_ws)
    local_ms = 1.0 + rank            # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, got_ws, device="cpu")
    q.put((got_rank, got_ws, ms, bench.job_throughput(10**9, got_ws, ms)))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == 2.0 for r in res)                 # max over ranks
    assert all(abs(r[3] - 2 * 1e9 / 2e-3 / 1e9) < 1e-9 for r in res)   # both ranks' bytes / slowest time


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_its_line():
    """Rank 0 of the reference arm: the CPU oracle on a bounded sample, one JSON line."""
    pytest.importorskip("scipy")
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "c1",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["unit"] == "GB/s"
