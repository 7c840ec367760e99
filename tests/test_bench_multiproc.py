"""bench.py's multi-process path on CPU (gloo, world size 2): replicas only.

Each rank runs the same workload on its own GPU; the only communication is
host-side: a barrier around the timed region and the max over ranks of the
timings. The reference arm prints on rank 0 only.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_env()
    dist = bench.dist_init(ws)
    try:
        bench.barrier(dist)
        got = bench.reduce_max([float(rank + 1), 10.0 - rank, 0.5 * rank], dist)
        q.put((rank, ws, r, local, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, local, got in res:
        assert ws == 2 and r == rank and local == rank
        assert got == [2.0, 10.0, 0.5]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init(1) is None
    assert bench.reduce_max([3.0, 1.0], None) == [3.0, 1.0]


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2")
    outs = []
    procs = []
    for rank in range(2):
        e = dict(env, RANK=str(rank), LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--steps", "1", "--warmup", "3", "--m", "1", "--cpu-stride", "64"],
            env=e, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, cwd=ROOT))
    for p in procs:
        out, err = p.communicate(timeout=600)
        assert p.returncode == 0, err
        outs.append(out.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["higher_is_better"] is False
