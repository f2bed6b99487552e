"""The multi-process path of bench.py on the CPU (gloo, world size 2).

Batches are independent problems, so ranks never exchange data: the only
cross-rank operations are the barrier and the max of the timed region, and
the whole-job rate sums every rank's units over the slowest rank's time.
"""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        dist.barrier()
        my_ms = 100.0 + 50.0 * rank                # rank 1 is the slow one
        mx = bench.max_over_ranks(my_ms, "cpu")
        rate = bench.whole_job_rate(1000, ws, 10, mx)
        out[rank] = (mx, rate, bench.rank_seed(2, rank))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    ws = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(ws, port, out), nprocs=ws, start_method="spawn")
    assert out[0][0] == out[1][0] == 150.0          # both ranks see the slowest time
    assert out[0][1] == out[1][1] == 1000 * 2 * 10 / 0.150
    assert out[0][2] is None and out[1][2] is not None   # different batches per rank


def test_single_process_helpers():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10, 1, 4, 2.0) == 10 * 4 / 0.002


def _run(cmd, env=None, timeout=600):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run(cmd, cwd=ROOT, env=e, capture_output=True, text=True, timeout=timeout)


def test_reference_arm_on_cpu():
    r = _run([sys.executable, "bench.py", "--impl", "reference", "--config", "1",
              "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    r = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
              "--master-addr", "127.0.0.1", f"--master-port={port}", "bench.py", "--impl",
              "reference", "--config", "1", "--steps", "3", "--warmup", "3"], timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2
