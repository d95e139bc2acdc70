"""The replicas path of bench.py (one process per GPU, no exchange on the data path) on CPU:
two gloo ranks report different step times; the job rate must come from the slowest rank."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [0.25 + 0.1 * rank, 0.30 + 0.05 * rank]       # rank 1 is the slower one
    agg = bench.aggregate_ranks(ms, dist, None)
    dist.barrier()
    out[rank] = agg
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == pytest.approx([0.35, 0.35])
    import bench
    assert bench.job_rate(world, 63, 0.35) == pytest.approx(2 * 63 / 0.35e-3)
    assert bench.aggregate_ranks([1.0, 2.0]) == [1.0, 2.0]


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference"])
    bench.main()  # rank 1: no work, no output
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_the_tiny_workload(capsys, monkeypatch):
    """The reference arm (the fp64 oracle on the host cores) prints one JSON line with the
    native arm's metric, unit and direction, the e2e object with zero copy bytes, and a
    cpu_baseline describing the run; it stops at the requested step count."""
    import json
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--workload", "1", "--steps", "2",
                                     "--warmup", "1"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == bench.UNIT
    assert j["higher_is_better"] is True and j["steps"] == 2 and j["value"] > 0
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
