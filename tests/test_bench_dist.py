"""Multi-process plumbing of bench.py on CPU (gloo, world size 2).

bench.py runs one process per GPU and reports the slowest rank's time; with
--impl reference only rank 0 runs the oracle and prints. These tests cover that
host logic without a GPU.
"""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    assert (w, r) == (world, rank)
    d = bench.maybe_init_dist(w, "gloo")
    # each rank's timed total; the job's time is the slowest rank's
    got = bench.max_over_ranks(10.0 + 5.0 * rank, d)
    out[rank] = got
    d.barrier()
    d.destroy_process_group()


def test_max_over_ranks_takes_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_needs_no_process_group():
    assert bench.maybe_init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_reference_arm_prints_one_line_from_rank_zero_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--config", "tiny16"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
