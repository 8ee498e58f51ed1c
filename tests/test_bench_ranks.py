"""The host side of bench.py's N > 1 path, on CPU: two gloo ranks on
127.0.0.1.  The path runs replicas (one per GPU, no data-path collective),
so what the ranks share is the timing: every rank must end with the slowest
rank's step time, the job's rate counts all ranks' bytes over that time, and
the reference arm does its work on rank 0 only."""
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, step_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(step_ms[rank], dist, device="cpu")
        out.put((rank, ms, bench.whole_job_gbs(world, 1_000_000_000, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world, step_ms):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, step_ms, out)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=180) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    return res


def test_every_rank_gets_the_slowest_step_time():
    res = _run(2, [2.5, 4.0])
    assert [r for r, _, _ in res] == [0, 1]
    assert all(ms == 4.0 for _, ms, _ in res)
    # two replicas of 1 GB each over the slowest rank's 4 ms
    assert all(abs(gbs - 2 * 1e9 / 4e-3 / 1e9) < 1e-9 for _, _, gbs in res)


def test_alone_the_value_is_kept_and_the_rate_is_one_ranks():
    assert bench.max_over_ranks(3.25, None) == 3.25
    assert bench.whole_job_gbs(1, 2_000_000_000, 2.0) == pytest.approx(1000.0)


def test_reference_arm_does_no_work_off_rank_0():
    class Args:
        steps, warmup, ref_frac, workload, layers = 2, 3, 0.0625, "stack52_m1", 52
    assert bench.run_reference(Args(), 1, 2) is None


def test_clock_sampler_parses_samples_and_cleans_up(tmp_path, monkeypatch):
    # a stand-in for nvidia-smi that prints three samples in the queried CSV
    # form (one of them with sw_power_cap active) and then waits to be stopped
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '0, 1950, 2070, 1399.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "echo '0, 2070, 2070, 950.3, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ.get('PATH', '')}")
    import time
    s = bench.ClockSampler(None)
    s.start()
    path = s.path
    time.sleep(0.5)
    got = s.stop()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not os.path.exists(path)


def test_reference_arm_line_has_the_contract_keys():
    # the reference arm times the fp64 oracle on a small row sample of one
    # layer; its JSON line carries the keys and units of the native line
    class Args:
        steps, warmup, ref_frac, workload, layers = 1, 3, 0.002, "stack52_m1", 52
    res = bench.run_reference(Args(), 0, 1)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in res, k
    assert res["impl"] == "reference" and res["unit"] == "GB/s" and res["higher_is_better"] is True
    assert res["value"] > 0 and res["steps"] == 1 and res["n_gpus"] == 1
    assert res["metric"] == bench.METRIC and res["config"]["workload"]
    cb = res["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == res["value"] and cb["cores"] >= 1 and cb["sample"]
    assert res["e2e"] == {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    import json
    json.dumps(res)
