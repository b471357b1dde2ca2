"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

Every rank runs its own replica; the timed region is bracketed by barriers
and the slowest rank's time is taken (max over ranks).  The reference arm
runs on rank 0 only.
"""
import os
import socket
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
    r, w, lr = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    mx = bench.reduce_max(10.0 + r, dist)
    bench.barrier(dist)
    ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(),
                              __import__("ssd_sequence_mixing_fwd_b300.inputs", fromlist=["x"])
                              .WORKLOADS["tiny_fp32"])
    dist.destroy_process_group()
    q.put((r, w, mx, ref is not None))


def test_two_rank_gloo_max_and_rank0_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[2] == 11.0 for r in res)           # max over ranks
    assert res[0][3] is True and res[1][3] is False  # reference arm on rank 0 only
