"""Host-side logic of bench.py that needs no GPU: byte accounting, the
max-over-ranks / sum-over-ranks aggregation (two gloo ranks on CPU), and the
reference arm's rank rule."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_step_bytes():
    kb = bench.kernel_bytes(8192, 8192)
    assert kb["scale2d"] == kb["copy2d"] == kb["affine"] == 8 * 8192 * 8192
    assert kb["rowsum"] == kb["rowmax_masked"] == 4 * 8192 * 8192 + 4 * 8192
    assert sum(kb.values()) == 2_416_017_408


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(1.25, 1000, 1) == (1.25, 1000)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank,) + bench.aggregate(1.0 + rank, 100 * (rank + 1), world))
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time and the bytes of all ranks
    assert got == [(0, 2.0, 300), (1, 2.0, 300)]


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args) is None
