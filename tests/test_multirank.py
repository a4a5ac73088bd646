"""Multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

The hot path shards by replication (every rank runs its own copy of the
workload on its own GPU, no collective on the data path), so what needs
covering with several processes is the host side: the rank/world discovery,
the barrier, the max-over-ranks timing reduction and the weak-scaling value,
and the reference arm's rule that only rank 0 works and prints.
"""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, local, w = bench.dist_info()
    bench.init_dist(w, "gloo")
    try:
        bench.barrier(w)
        t_max = bench.max_over_ranks(times[r], w)
        value = bench.weak_scaling_value(1000.0, w, t_max)   # 1000 units per rank
        bench.barrier(w)
        out.put((r, local, w, t_max, value))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_weak_scaling():
    world = 2
    times = [0.25, 0.75]                     # rank 1 is the slow one
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    res = sorted(out.get(timeout=5) for _ in range(world))
    for r, (rank, local, w, t_max, value) in enumerate(res):
        assert (rank, local, w) == (r, r, world)
        # every rank sees the slowest rank's time ...
        assert t_max == max(times)
        # ... and the whole-job throughput counts every rank's units over it
        assert value == pytest.approx(1000.0 * world / max(times))


def test_single_rank_helpers_need_no_process_group(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_info() == (0, 0, 1)
    bench.init_dist(1, "gloo")                     # no process group for one rank
    assert not torch.distributed.is_initialized()
    bench.barrier(1)
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.weak_scaling_value(10.0, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    """Under torchrun only rank 0 times the oracle and prints its line."""
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    def _no_oracle(*a, **k):
        raise AssertionError("rank 1 must not run the oracle")

    monkeypatch.setattr(bench, "time_oracle", _no_oracle)
    monkeypatch.setattr(bench, "oracle_sample", _no_oracle)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert rc in (0, None)
    assert buf.getvalue() == ""


def test_reference_arm_prints_the_contract_line(monkeypatch):
    """``bench.py --impl reference`` (rank 0, one process) times the oracle on
    the host cores and prints one JSON line with the contract's keys: the
    arm's name, the metric and unit, a cpu_baseline describing the run, and
    an e2e object with no host/device bytes."""
    import json
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                         "--warmup", "3"])
    assert rc in (0, None)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
