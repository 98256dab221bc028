"""The bench's host logic on CPU: max over ranks of the per-rank step times (gloo, two
processes), whole-job throughput, the reference arm's rank > 0 exit and its JSON line,
and the clock record's window."""

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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured step r+1 ms and e2e 10(r+1) ms
    got = bench.max_over_ranks([1.0 + rank, 10.0 * (1 + rank)], world)
    q.put((rank, got, bench.job_throughput(world, 8, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, thr in res:
        assert got == [2.0, 20.0]                  # every rank sees the slowest replica
        assert thr == pytest.approx(2 * 8 / 2e-3)  # 16 queries per 2 ms


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.5, 7.0], 1) == [3.5, 7.0]
    assert bench.job_throughput(1, 8, 0.5) == pytest.approx(16000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_clock_samples_are_taken_from_the_timed_region():
    """The clock record keeps the nvidia-smi samples stamped inside the timed region (a
    throttle reason seen only outside it is not reported), and falls back to every
    sample when none falls inside."""
    import datetime
    import time
    import bench

    now = datetime.datetime.now()
    inside = now.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    outside = (now - datetime.timedelta(seconds=30)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    text = (inside + ", 0, 2070 MHz, 2070 MHz, 900.00 W, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            + outside + ", 0, 1200 MHz, 2070 MHz, 300.00 W, 0x0, Not Active, Not Active, Active, Not Active\n")

    class FakeSmi:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return text, ""

    c = bench.ClockSampler("0")
    c.proc = FakeSmi()
    c.t0, c.t1 = time.time() - 5, time.time() + 5
    got = c.stop()
    assert got["window"] == "timed region" and got["samples"] == 1
    assert got["sm_mhz"] == 2070.0 and got["reasons"] == []
    c = bench.ClockSampler("0")
    c.proc = FakeSmi()
    c.t0, c.t1 = time.time() + 100, time.time() + 101   # a region no sample falls in
    got = c.stop()
    assert got["window"] == "around the timed region" and got["samples"] == 2
    assert got["reasons"] == ["sw_thermal_slowdown"]


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line with
    the benchmark's metric and unit, its own cpu_baseline and a zero-copy e2e object."""
    import json
    import bench
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "queries/s"
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "queries/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert "workload" in line["config"]
