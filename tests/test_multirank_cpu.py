"""Host logic of the multi-GPU (replicas) bench path, on CPU.

Each rank runs its own layers (the path shards by independent layers, with no
data-path collective); the job's time is the slowest rank's and its units are
the sum over ranks.  Two gloo ranks stand in for two GPUs.  The reference arm
runs on rank 0 only: the other ranks exit without work.
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


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        ms = [12.0, 15.5][rank]
        units = [1.0e6, 3.0e6][rank]
        t, u = bench.job_time_and_units(ms, units, ws, torch.device("cpu"))
        q.put((rank, env, t, u))
    finally:
        dist.destroy_process_group()


def test_two_rank_job_time_is_max_and_units_are_summed():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, env, t, u in got:
        assert env == (2, rank, rank)
        assert t == 15.5 and u == 4.0e6


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_and_units(3.0, 7.0, 1, torch.device("cpu")) == (3.0, 7.0)


def _bench(env_extra, *args):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_runs_on_rank_zero_only():
    args = ("--impl", "reference", "--workload", "tiny_decode", "--steps", "1", "--warmup", "1")
    r1 = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, *args)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _bench({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, *args)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
