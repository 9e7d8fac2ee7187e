"""Multi-rank logic of bench.py on CPU: two gloo ranks (127.0.0.1), each with
its own step time; every rank must see the slowest one, and the whole-job
value must count both replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(ms[rank], "cpu")
        q.put((rank, got, bench.whole_job_tflops(world, 2e12, got)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ms = [18.5, 21.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, tflops in res:
        assert got == pytest.approx(21.25)
        assert tflops == pytest.approx(2 * 2e12 / 21.25e-3 / 1e12)


def test_single_process_values_pass_through():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)


def _fake_smi(real_popen, line):
    """A stand-in for `nvidia-smi -lms`: prints one CSV sample line every
    50 ms until it is terminated."""
    import sys

    def popen(cmd, **kw):
        code = f"import time\nwhile True:\n print({line!r}, flush=True)\n time.sleep(0.05)"
        return real_popen([sys.executable, "-c", code], **kw)
    return popen


def test_clock_sampler_parses_samples_and_ends_its_child(monkeypatch):
    import subprocess
    import time
    line = "0, 1980, 2070, 910.5, 0x4, Not Active, Not Active, Not Active, Active"
    monkeypatch.setattr(bench.subprocess, "Popen", _fake_smi(subprocess.Popen, line))
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.3)
    got = c.stop()
    assert c.proc.poll() is not None
    assert got["sm_mhz"] == 1980.0 and got["sm_max_mhz"] == 2070.0
    assert got["samples"] >= 1 and got["reasons"] == ["sw_power_cap"]


def test_clock_sampler_child_ends_even_without_stop(monkeypatch):
    """The sampler registers its own end at interpreter exit, so a timed
    region that raises leaves no nvidia-smi loop behind; ending twice is
    harmless."""
    import subprocess
    import time
    monkeypatch.setattr(bench.subprocess, "Popen",
                        _fake_smi(subprocess.Popen, "0, 1, 2, 3, 0x0, a, b, c, d"))
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.1)
    assert c.proc.poll() is None
    c._end()          # what the exit hook runs
    c._end()
    assert c.proc.poll() is not None
    got = c.stop()    # stop after the end still reads what was sampled
    assert got["sm_mhz"] == 1.0 and got["reasons"] == []


def test_peak_follows_the_clock_record():
    """The bf16 denominator is the burst peak unless the timed region lasted
    seconds with the power cap active, then the sustained one."""
    pk = {"bf16": 1914.7, "bf16_sustained": 1693.2, "hbm": 6783.8, "source": "measured"}
    row = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    short_capped = bench.ClockSampler.summarise([row.format(sm=1800, cap="Active").split(",")] * 4)
    assert short_capped["power_cap_samples"] == 4
    long_free = bench.ClockSampler.summarise([row.format(sm=2070, cap="Not Active").split(",")] * 9)
    assert long_free["reasons"] == [] and long_free["sm_mhz"] == 2070.0
    assert bench.choose_bf16_peak(pk, long_free, 20.0)[0] == 1914.7
    assert bench.choose_bf16_peak(pk, short_capped, 0.4)[0] == 1914.7
    assert bench.choose_bf16_peak(pk, short_capped, 20.0)[0] == 1693.2
    assert bench.choose_bf16_peak(pk, None, 20.0)[0] == 1914.7
    fr = bench.peak_fractions(957.35, pk)
    assert fr["of_burst"] == pytest.approx(0.5) and fr["of_sustained"] > 0.5


def test_traffic_records_are_keyed_by_kernel_workload_and_source(tmp_path, monkeypatch):
    import json
    rec = tmp_path / "dram_traffic.json"
    sha = bench.source_hash(bench.BWD_KERNEL_SOURCES)
    rec.write_text(json.dumps({"records": [
        {"kernel": "bwd_kernel", "workload": "long", "dram_bytes_per_launch": 123,
         "kernel_source_sha256": sha},
        {"kernel": "bwd_kernel", "workload": "dense14b", "dram_bytes_per_launch": 7,
         "kernel_source_sha256": "0" * 64}]}))
    monkeypatch.setattr(bench, "TRAFFIC_RECORDS", str(rec))
    assert bench.recorded_traffic("long") == 123
    assert bench.recorded_traffic("dense14b") is None      # kernel changed since
    assert bench.recorded_traffic("drafter") is None       # never captured
