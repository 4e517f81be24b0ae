"""The multi-rank path of bench.py on the CPU: ranks are replicas (each
verifies its own batch, no exchange on the data path), so what N > 1 adds is
host logic -- the slowest rank's time taken by an all-reduce, the whole-job
rate, and rank 0 alone printing.  Exercised here with two gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        out.put((rank, slowest, bench.whole_job_rate(world, 100, slowest)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_whole_job_rate_two_gloo_ranks():
    times = [12.5, 20.0]  # ms of each rank's timed region
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in got:
        assert slowest == 20.0, (rank, slowest)         # every rank sees the slowest time
        assert rate == pytest.approx(2 * 100 / 0.020)   # both ranks' steps over that time


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.0, 1, torch.device("cpu")) == 7.0
    assert bench.whole_job_rate(1, 50, 250.0) == pytest.approx(200.0)


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference with two ranks: rank 0 times the oracle and
    prints one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    # ms_per_step is the time of one timed (sampled) step, value is in full
    # steps/s: the sample is sample_fraction_of_step of a step
    frac = d["sample_fraction_of_step"]
    assert 0 < frac <= 1
    assert d["ms_per_step"] * d["value"] == pytest.approx(1e3 * frac, rel=1e-6)
    cb, e2e = d["cpu_baseline"], d["e2e"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]
