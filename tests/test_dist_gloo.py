"""The benchmark's multi-rank bookkeeping on CPU with gloo, world size 2:
time is the max over ranks, bytes are summed, the reference arm runs on
rank 0 only.  (The GPU path itself shards nothing: ranks are replicas.)"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    bench.dist_init("gloo")
    t = bench.max_over_ranks(1.5 + rank)         # rank 1 is the slow one
    b = bench.sum_over_ranks(100.0 * (rank + 1))
    bench.barrier()
    q.put((rank, t, b))
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5, 300.0), (1, 2.5, 300.0)]


def _ref_worker(rank, world, port, q):
    import contextlib
    import io
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                    "--warmup", "1", "--gpus", str(world)])
    q.put((rank, buf.getvalue()))


def test_reference_arm_prints_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    out = dict(q.get(timeout=10) for _ in range(2))
    import json
    line = json.loads(out[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert out[1].strip() == ""
