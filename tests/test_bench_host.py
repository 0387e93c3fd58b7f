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


def test_link_floor_takes_the_slowest_leg():
    link = {"h2d_GBps": 200.0, "d2h_GBps": 100.0, "both_GBps": 250.0}
    # 1 GB each way: the download leg binds (10 ms against 8 ms for both at once)
    assert bench.link_floor_s(1e9, 1e9, link) == pytest.approx(1e9 / 100e9)
    # download-light: the upload leg binds
    assert bench.link_floor_s(4e9, 1e8, link) == pytest.approx(4e9 / 200e9)
    # balanced and a slow two-way rate: the shared link binds
    slow = dict(link, both_GBps=120.0)
    assert bench.link_floor_s(1e9, 1e9, slow) == pytest.approx(2e9 / 120e9)


def _cfg_row(config, us, us_clean, target):
    return {"config": config, "target": target, "lone": {"us": us, "frac": 1.0 / us},
            "lone_clean": {"us": us_clean, "frac": 1.0 / us_clean},
            "target_met": {} if target is not None else None}


def test_attach_floors_compares_with_the_same_config_floor():
    rows = {
        "C3_copy2d_ragged": _cfg_row("C3", 12.5, 8.2, 0.75),
        "C4_rowsum": _cfg_row("C4", 17.06, 16.38, 0.85),
        "C4_colsum_auto": _cfg_row("C4", 19.12, 18.43, 0.70),
        "C5_rowmax_masked": _cfg_row("C5", 13.0, 12.3, None),
        "C3_floor_memcpy": _cfg_row("C3", 16.03, 12.29, None),
        "C4_floor_read": _cfg_row("C4", 17.06, 16.38, None),
    }
    bench.attach_floors(rows)
    assert rows["C3_copy2d_ragged"]["floor"]["entry"] == "C3_floor_memcpy"
    assert rows["C3_copy2d_ragged"]["floor"]["lone_vs_floor"] == round(12.5 / 16.03, 3)
    assert rows["C3_copy2d_ragged"]["target_met"]["lone_within_5pct_of_floor"] is True
    assert rows["C4_rowsum"]["floor"]["lone_vs_floor"] == 1.0
    assert rows["C4_rowsum"]["target_met"]["lone_within_5pct_of_floor"] is True
    assert rows["C4_colsum_auto"]["floor"]["lone_clean_vs_floor"] == round(18.43 / 16.38, 3)
    assert rows["C4_colsum_auto"]["target_met"]["lone_within_5pct_of_floor"] is False
    # an untargeted row gets the comparison but no verdict; the floors none
    rows["C5_floor_read"] = _cfg_row("C5", 12.0, 11.0, None)
    bench.attach_floors(rows)
    assert rows["C5_rowmax_masked"]["floor"]["lone_vs_floor"] == round(13.0 / 12.0, 3)
    assert rows["C5_rowmax_masked"]["target_met"] is None
    for k in ("C3_floor_memcpy", "C4_floor_read", "C5_floor_read"):
        assert "floor" not in rows[k]
    # the column sums also meet the fixed-share read; no other row does
    rows["C4_floor_fixed_share"] = _cfg_row("C4", 18.0, 17.0, None)
    bench.attach_floors(rows)
    assert rows["C4_colsum_auto"]["floor_fixed_share"]["lone_vs_floor"] == round(19.12 / 18.0, 3)
    assert "floor_fixed_share" not in rows["C4_rowsum"]
    assert "floor" not in rows["C4_floor_fixed_share"]


def test_every_floor_names_a_config_entry():
    keys = {e[0]: e[1] for e in bench.CONFIG_ENTRIES}
    for cfg, fk in bench.FLOOR_OF.items():
        assert keys.get(fk) == cfg
    for row, fk in bench.FIXED_SHARE_FLOOR_OF.items():
        assert keys.get(row) == keys.get(fk) and keys.get(fk) is not None
