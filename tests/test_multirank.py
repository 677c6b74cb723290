"""The multi-process path of bench.py on CPU (gloo, world size 2).

The quantized Muon step does not shard across GPUs here ("replicas only"):
every rank runs its own copy of the workload and the job's time is the
slowest rank's.  These tests run the bench's rank helpers in two gloo
processes and the CPU-oracle leg on a small sample.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_info()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(world)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        v = bench.job_throughput(1_000_000, 4, world, t)
        out.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's 15 ms; 2 replicas x 1M params x 4 steps in 15 ms
    assert [r[1] for r in res] == [15.0, 15.0]
    assert all(abs(r[2] - 2 * 1e6 * 4 / 0.015 / 1e6) < 1e-6 for r in res)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(872_415_232, 10, 1, 1000.0) == pytest.approx(8724.15232)


def test_oracle_sample_leg():
    o = bench.oracle_sample(workloads.get(1), steps=2, warmup=1)
    assert o["value"] > 0 and o["cores"] >= 1 and "512x512" in o["sample"]
    assert o["steps"] == 2 and o["ms_per_step"] > 0 and o["extrapolated"] is True
    assert o["single_core"] is None or 0 < o["single_core"]


def test_executed_flop_count_of_the_syrk_schedule():
    # 256 x 256 tiles, symmetric products on and above the diagonal: on the
    # MuonBP workload's block set 1.357e13 FLOPs per call, full set 6.05e13
    w = workloads.get(4)
    assert abs(bench.step_ns_executed(w, False) - 1.3572e13) / 1.3572e13 < 1e-3
    assert abs(bench.step_ns_executed(w, True) - 6.0527e13) / 6.0527e13 < 1e-3
    # one 256 x 256 tile per product at m = n = 256: 3 x 2 x 256^3 per iteration
    assert bench.ns_executed_flops_of(256, 256, 1) == 3 * 2.0 * 256 ** 3


def test_step_flop_count_matches_page_formula():
    w = workloads.get(4)
    full = bench.step_ns_flops(w, True)
    block = bench.step_ns_flops(w, False)
    assert abs(full - 8.324e13) / 8.324e13 < 1e-3      # 2(2nm^2+m^3) x 5 over the 28 matrices
    assert abs(block - 1.705e13) / 1.705e13 < 1e-3     # the same over 224 tiles of 1x8 columns


def test_reference_arm_prints_the_contract_line():
    # `bench.py --impl reference` (the CPU oracle arm) prints one JSON line
    # with the keys of the benchmark contract, on the CPU, without a GPU
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1", "--steps", "2",
                        "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "Mparams/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["scaling"] == "weak"
    assert d["extrapolated"] is True   # value: the workload rate from the timed sample steps
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "single_512"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "Mparams/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_clock_sampler_summarises_nvidia_smi_lines():
    # the clocks record of the bench line from nvidia-smi's CSV rows (index,
    # sm, max sm, power, active, hw_slowdown, hw_thermal, sw_thermal,
    # sw_power_cap): median SM clock under load, the maximum, and every
    # throttle reason seen active
    class _Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.lines = ["0, 1965, 2070, 1100.5, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 1710, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 1800, 2070, 1250.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "[N/A] garbled line",
               "0, 1500, 2070, 1400.0, 0x40, Not Active, Active, Not Active, Not Active"]
    c = s.stop()
    assert c["samples"] == 4 and c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == 1755.0                                   # median of 1965, 1710, 1800, 1500
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]
