"""The multi-GPU path of bench.py is replicas: one independent layer per rank, no data-path
collective, a barrier around the timed region, the slowest rank's time, and the whole job's
tokens. Its host logic runs here as world_size-2 gloo ranks on CPU; the reference arm under
torchrun prints one line from rank 0 while the other rank exits without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")   # rank 1 is the slow one
        out[rank] = (ms, bench.job_tokens_per_s(world, 8192, 4, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # spawn, never fork, from a process with threads
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                               # every rank sees the same job time
    ms, value = res[0]
    assert ms == 15.0                                     # the slowest rank's
    assert value == pytest.approx(2 * 8192 * 4 / 15e-3)   # both ranks' tokens


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(1, 100, 10, 1000.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny_f32", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-tokens", "4"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
