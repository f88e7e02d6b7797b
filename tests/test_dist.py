"""The benchmark's multi-process path on CPU (gloo, two ranks).

The method shards only as independent replicas: every rank runs the whole
workload on its own GPU and the ranks exchange nothing but the timing (a
barrier around the timed region and the maximum elapsed time over ranks).
These tests run that exchange with two gloo ranks, and the reference arm
launched through torch.distributed.run, where rank 0 alone prints one line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.dist_barrier(w)
    # each rank reports its own elapsed time; every rank must see the maximum
    out[rank] = bench.dist_max(10.0 + 5.0 * rank, w)
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_gloo_max_over_ranks():
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world,
                           start_method="spawn", join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


@pytest.mark.slow
def test_reference_arm_under_torchrun():
    import oracle
    oracle.num_threads()  # builds the oracle library before the ranks start
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 1
    assert rec["warmup"] == 3 and rec["value"] > 0 and rec["unit"] == "TFLOP/s"
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
