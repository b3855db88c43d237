"""Multi-process (replica) paths of bench.py on the CPU: gloo, world size 2.

The decode step does not shard (the pages make tensor parallelism a non-goal),
so N GPUs run N independent replicas; the only cross-rank steps are the
barrier, the max over ranks of the timed region and rank 0's single JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 20.0][rank]  # rank 1 is the slower replica
    got = bench.max_over_ranks(ms, dist)
    out[rank] = (got, bench.job_rate(world, 128, got))
    dist.barrier()
    dist.destroy_process_group()


def test_timed_region_is_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as man:  # no fork of a threaded process
        out = man.dict()
        mp.spawn(_reduce_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # every rank sees the slowest replica's 20 ms; the job did 2 x 128 tokens in it
    assert res[0] == res[1] == (20.0, 2 * 128 / 0.020)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(7.0, None) == 7.0
    assert bench.job_rate(1, 64, 500.0) == 128.0


def test_reference_arm_under_torchrun_prints_one_line():
    # the reference arm (the oracle on the host cores) under torchrun: rank 0
    # alone runs and prints, the other rank exits 0 without work
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "0",
           "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
