"""Host logic of bench.py for more than one rank, on CPU with the gloo backend.

The path has no exchange step: each rank runs its own replica of the workload,
the timing is the maximum over ranks, and the whole-job rate counts every
rank's tokens. These tests run that logic as two real processes.
"""
from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        # rank r took (r + 1) ms for the whole step and (10 - r) ms for one stage
        mx = bench.max_over_ranks([rank + 1.0, 10.0 - rank])
        rate = bench.whole_job_rate(4096, ws, mx[0])
        # the reference arm: only rank 0 runs and prints
        args = type("A", (), {"workload": "tiny", "seed": 0, "steps": 0, "warmup": 0})()
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(args)
        results[rank] = (ws, r, local, mx, rate, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank, (ws, r, local, mx, rate, printed) in res.items():
        assert (ws, r, local) == (2, rank, rank)
        assert mx == [2.0, 10.0]                      # maximum over both ranks, element by element
        assert rate == pytest.approx(2 * 4096 / 2e-3)  # both ranks' tokens over the slowest rank's time
    assert res[1][5] == ""                            # rank 1 of the reference arm prints nothing


def test_single_process_helpers():
    assert bench.max_over_ranks([1.5, 2]) == [1.5, 2.0]
    assert bench.whole_job_rate(1000, 1, 2.0) == pytest.approx(5e5)


def test_algorithmic_bytes_fixed_workload():
    from chunked_gated_delta_02_gb300.workloads import named
    w = named("fixed")
    inp = {"B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V, "N": w.B, "initial_state": None}
    th = 2 * 2048 * 32
    assert bench.algorithmic_bytes(inp, with_state=False) == th * 1282
    assert bench.algorithmic_bytes(inp) == th * 1282 + 2 * 32 * 128 * 128 * 4


def test_reference_arm_json_line(monkeypatch):
    """The reference arm's line (rank 0, one process): the oracle timed on the host cores, with the
    keys the driver reads. The sample is shortened for the test."""
    import json
    orig = bench.cpu_baseline
    monkeypatch.setattr(bench, "cpu_baseline", lambda inp, target_s=8.0: orig(inp, target_s=0.2))
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    args = type("A", (), {"workload": "tiny", "seed": 0, "steps": 1, "warmup": 0})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True and line["steps"] == 1
    assert line["config"]["workload"].startswith("tiny")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_each_kernel_is_credited_with_its_own_bytes():
    """The prep kernel is credited with q, k, g and beta (770 B per token-head at K = 128), the
    recurrence kernel with v, o and the state; together they are the path's algorithmic bytes."""
    inp = dict(B=2, T=2048, H=32, K=128, V=128, N=2, initial_state=None)
    th = 2 * 2048 * 32
    ab = bench.kernel_algorithmic_bytes(inp)
    assert ab["prep"] == th * 770
    assert ab["recurrence"] == th * 512 + 2 * 32 * 128 * 128 * 4
    assert ab["prep"] + ab["recurrence"] == bench.algorithmic_bytes(inp) == th * 1282 + 2 * 32 * 128 * 128 * 4
    roofs = bench.kernel_rooflines(inp, 0.0907, 0.0581, 6680.8, "test", "no-such-workload")
    assert roofs[0]["kernel"].startswith("prep")
    assert abs(roofs[0]["frac"] - th * 770 / 90.7e-6 / 1e9 / 6680.8) < 1e-9
    assert abs(roofs[0]["frac"] - 0.1666) < 1e-3
    assert roofs[0]["traffic"] is None and roofs[0]["traffic_over_algorithmic"] is None


def test_batch_and_head_overrides(monkeypatch):
    """--batch and --heads resize a fixed-length workload and keep everything else; a varlen
    workload refuses --batch."""
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "large_batch", "--batch", "16", "--heads", "8"])
    w = bench.workload_of(bench.parse())
    assert (w.B, w.T, w.H, w.K, w.V, w.lower_bound) == (16, 512, 8, 128, 128, -5.0)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "varlen", "--batch", "16"])
    with pytest.raises(SystemExit):
        bench.workload_of(bench.parse())
