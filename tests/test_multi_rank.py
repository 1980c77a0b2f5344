"""Host-side logic of the N > 1 path, on CPU with gloo (world size 2).

Encode/apply need no collective; with N GPUs bench.py runs N independent
replicas and only reduces timings (max over ranks) and work (sum over ranks).
The reference arm runs on rank 0 alone; other ranks exit without work.
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    mx = bench.max_over_ranks(float(rank + 1) * 10.0, True)
    sm = bench.sum_over_ranks(float(rank + 1), True)
    bench.barrier(True)
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_rank_reductions_with_gloo():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == (20.0, 3.0)
    assert out[1] == (20.0, 3.0)


def test_single_rank_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, False) == 1.5
    assert bench.sum_over_ranks(2.5, False) == 2.5


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--config", "1", "--steps", "1", "--warmup", "0", "--cpu-sample-params", "1e5"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
