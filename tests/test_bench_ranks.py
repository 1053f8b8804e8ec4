"""bench.py with more than one rank, on CPU: two gloo ranks, one process each.

With N GPUs the bench runs one process per GPU, each selecting from its own
row (weak scaling, no collective on the data path); the ranks meet only at
barriers and in the max-reduction of their timed regions, and the job's value
counts every rank's elements over the slowest rank's time.  These tests run
that host logic with the gloo backend, and check that the reference arm's
other ranks leave without work."""
import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, ws, "cpu")
        q.put((rank, env, slowest, bench.job_gelems(1 << 30, 20, ws, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r[1] for r in res] == [(2, 0, 0), (2, 1, 1)]
    assert [r[2] for r in res] == [15.0, 15.0]  # both ranks see the slower rank's 15 ms
    assert res[0][3] == res[1][3] == pytest.approx(2 * 20 * 2**30 / 0.015 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_gelems(1 << 30, 10, 1, 1000.0) == pytest.approx(10 * 2**30 / 1e9)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(gpus=2, steps=3, warmup=3, n=1 << 30, k=1024)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_workload_names_and_l2_note():
    assert bench.workload_name("normal", 1 << 30, 1024) == "normal_2^30_k1024"
    assert bench.workload_name("levels16", 1 << 28, 4096) == "levels16_2^28_k4096"
    assert bench.workload_name("sae", 50_331_648, 131_072) == "sae_50331648_k131072"
    assert bench.l2_note(1 << 30).startswith("input 4295 MB > L2")
    assert "hot-cache" in bench.l2_note(1 << 22)
    assert set(bench.INPUTS) >= {"normal", "uniform", "pareto", "ulps_below_one", "levels16", "sae"}


def test_reference_arm_prints_its_line():
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the contract's keys, without a GPU."""
    import json
    import subprocess
    import sys

    out = subprocess.run([sys.executable, str(bench.ROOT / "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "Gelem/s"
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["n"] == bench.REF_SAMPLE_ELEMS and d["config"]["workload"] == "normal_2^30_k1024"
    assert d["cpu_baseline"]["cores"] == bench.host_cores()


def test_config_entry_and_binomial_bound():
    sts = [{"attempts": 1, "aux_bytes": 10, "path": 0}, {"attempts": 3, "aux_bytes": 30, "path": 1}]
    e = bench.config_entry(1 << 30, 0.5, sts, 6800.0)
    assert e["retries"] == 2 and e["aux_bytes"] == 30 and e["paths"] == [0, 1]
    assert e["hbm_gbs"] == pytest.approx(4 * 2**30 / 0.5e-3 / 1e9, abs=0.1)
    assert e["hbm_frac_of_8TBs"] == pytest.approx(e["hbm_gbs"] / 8000, abs=1e-3)
    # P(Binomial(10^4, 10^-3) <= 18) >= 0.99 > P(... <= 17): the bound the retry run is read against.
    assert bench.binom_upper(10_000, 1e-3) == 18
