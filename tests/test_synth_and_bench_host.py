"""CPU checks of the seeded generators and of bench.py's host logic, including
the multi-rank aggregation on a world of two gloo processes."""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from mhc_hyper_connection_hc_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_generators_are_deterministic_and_seed_dependent():
    a = synth.uniform(123, 1000, -1, 1)
    b = synth.uniform(123, 1000, -1, 1)
    c = synth.uniform(124, 1000, -1, 1)
    assert a.dtype == np.float32 and np.array_equal(a, b) and not np.array_equal(a, c)
    assert a.min() >= -1 and a.max() < 1
    # chunked generation gives the same stream as one call
    big = synth.uniform(5, (1 << 22) + 17, 0, 1)
    assert np.array_equal(big[-17:], synth.uniform(5, (1 << 22) + 17, 0, 1)[-17:])
    assert np.array_equal(synth._u53(5, (1 << 22), 17), synth._u53(5, 0, (1 << 22) + 17)[-17:])


def test_generator_distributions():
    u = synth.uniform(9, 200000, 0.5, 1.5).astype(np.float64)
    assert abs(u.mean() - 1.0) < 0.01 and abs(u.var() - 1 / 12) < 0.003
    n = synth.normal(10, 200000, 0.0, 2.0).astype(np.float64)
    assert abs(n.mean()) < 0.02 and abs(n.std() - 2.0) < 0.02


def test_workload_shapes():
    w = synth.WORKLOADS[3]
    assert (w.T, w.s, w.d, w.R, w.K) == (4096, 4, 4096, 24, 16384)
    w5 = synth.WORKLOADS[5]
    assert (w5.s, w5.d, w5.R) == (8, 7168, 80) and w5.x_dist == "normal"
    inp = synth.site_inputs(1, 2, 4, 64)
    assert inp["x"].shape == (2, 4, 64) and inp["fn_w"].shape == (24, 256)
    assert inp["scale"].shape == (3,) and inp["base"].shape == (24,) and inp["f"].shape == (2, 64)
    # fn_w ~ N(0, 1/(s*d)) as a variance
    w_ = synth.site_params(3, 0, 4, 4096)[0].astype(np.float64)
    assert abs(w_.std() * np.sqrt(16384) - 1.0) < 0.01


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _agg_worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    t, u = bench.aggregate(1.0 + rank, 100.0 * (rank + 1))
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_bench_aggregation_two_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_agg_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, t, u in res:
        assert t == 2.0 and u == 300.0     # slowest rank's time, all ranks' tokens


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--ref-tokens", "4"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_sampler_keeps_the_samples_inside_the_measurement_region(tmp_path):
    """bench.py's clock summary: the median SM clock and the throttle reasons of the
    samples whose timestamps fall inside the measurement region (the timed steps and the
    per-kernel rounds after them), with the counts in the timed and the measurement
    region; sm_mhz is null when no sample falls inside."""
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    rows = [  # seconds after t0, SM MHz, hw_slowdown, sw_power_cap
        (-0.3, 1000, "Not Active", "Not Active"),
        (0.1, 2070, "Not Active", "Active"),
        (0.2, 2040, "Not Active", "Not Active"),
        (0.3, 2070, "Not Active", "Not Active"),
        (0.9, 500, "Active", "Not Active"),
    ]
    path = tmp_path / "clocks.csv"
    with open(path, "w") as fh:
        for dt, mhz, hw, cap in rows:
            stamp = (t0 + datetime.timedelta(seconds=dt)).strftime(bench.ClockSampler.STAMP)[:-3]
            fh.write(f"{stamp}, 0, {mhz}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, {cap}\n")

    def summary(start, end, region_end=None):
        cs = bench.ClockSampler(0)
        cs.proc, cs.path = object(), str(path)
        cs.t0 = t0 + datetime.timedelta(seconds=start)
        cs.t1 = t0 + datetime.timedelta(seconds=end)
        cs.t2 = None if region_end is None else t0 + datetime.timedelta(seconds=region_end)
        import shutil
        keep = str(path) + ".keep"
        shutil.copy(path, keep)
        try:
            return cs.summary()
        finally:
            shutil.move(keep, path)

    s = summary(0.0, 0.15, 0.5)
    assert s["samples"] == 5 and s["samples_in_timed_region"] == 1
    assert s["samples_in_measurement_region"] == 3
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]            # the hw_slowdown sample lies outside
    s = summary(0.0, 0.5)                              # no rounds: the timed region alone
    assert s["samples_in_measurement_region"] == 3 and s["sm_mhz"] == 2070
    s = summary(5.0, 6.0)                              # no sample inside: no clock reported
    assert s["samples_in_timed_region"] == 0 and s["sm_mhz"] is None and s["reasons"] == []
