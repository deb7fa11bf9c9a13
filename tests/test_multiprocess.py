"""The N > 1 launch path of bench.py on CPU with the gloo backend.

Multi-GPU here means replicas: every rank runs the whole hot path on its own
GPU and its own inputs, and only the timing and the row counts cross ranks
(max of the elapsed times, sum of the attended rows).  These tests run two
ranks as processes on the host: the rank reductions and barrier the GPU arm
uses, and the reference arm (the oracle), where rank 0 alone runs and prints
one JSON line and the other ranks exit 0 without work.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    bench = _load_bench()
    r, w, local = bench.dist_init("gloo")
    import torch
    dev = torch.device("cpu")
    mx = bench.max_over_ranks(1.5 + r, w, dev)
    sm = bench.sum_over_ranks(10.0 * (r + 1), w, dev)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, local, mx, sm))


def test_rank_reductions_two_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    for r, w, local, mx, sm in res:
        assert w == 2 and local == r
        assert mx == 2.5            # max over ranks of the elapsed time
        assert sm == 30.0           # sum over ranks of the rows processed


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "csa_decode"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout            # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
