"""The bench's multi-rank host logic with two gloo ranks on CPU: the slowest
rank's time is what every rank sees, whole-job throughput counts every rank's
replica, and the reference arm prints one line, from rank 0, with our arm's
config."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    w, r, local = bench.dist_setup()
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + r * 0.5, w)  # rank 1 is the slow one
    q.put((r, w, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 1.5), (1, 2, 1.5)]


def test_replica_throughput_counts_every_rank():
    import bench
    assert bench.replica_throughput(1e12, 10, 1, 2.0) == pytest.approx(5.0)
    assert bench.replica_throughput(1e12, 10, 4, 2.0) == pytest.approx(20.0)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def _reference_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import contextlib
    import io
    import json
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "tiny_f32", "--gpus", str(world),
                         "--steps", "1", "--warmup", "3", "--ref-seconds", "1"])
    lines = [json.loads(x) for x in buf.getvalue().splitlines() if x.startswith("{")]
    q.put((rank, rc, lines))


def test_reference_arm_under_two_ranks_prints_once_with_our_config():
    """Under torchrun the reference arm runs on rank 0 alone; its config is
    the one our arm prints at the same world size."""
    import bench
    from tiled_online_softmax_02_gb300.inputs import make_inputs
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reference_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rc0, lines0), (r1, rc1, lines1) = got
    assert (r0, r1) == (0, 1) and rc0 == 0 and rc1 == 0
    assert lines1 == [] and len(lines0) == 1
    w = bench.ALL_WORKLOADS["tiny_f32"]
    flops, excl = bench.flops_of(w, make_inputs(w))
    assert lines0[0]["impl"] == "reference"
    assert lines0[0]["config"] == bench.workload_config(w, flops, excl, 2)
