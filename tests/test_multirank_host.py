"""Host-side multi-rank logic of bench.py on CPU with the gloo backend
(world size 2): the timing barrier, the max-over-ranks reduction of the
elapsed time, and the reference arm running on rank 0 only.  Heads are
independent, so the data path has no collective; only this timing logic
crosses ranks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_setup()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    # each rank reports a different elapsed time; every rank must see the max
    got = bench.max_over_ranks(10.0 + 5.0 * rank, ws)
    out[rank] = got
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def _ref_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import contextlib
    import io
    import bench
    from certified_fixed_stabilizer_gb300.workloads import WORKLOADS

    class A:
        steps, warmup, gpus, variant = 1, 0, world, "auto"
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(A, WORKLOADS["tiny"], WORKLOADS["tiny"].H)
    out[rank] = buf.getvalue()


def test_reference_arm_prints_on_rank0_only_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_ref_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    assert out[1] == ""
    import json
    line = json.loads(out[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
