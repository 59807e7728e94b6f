"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank of a replicated run times its own steps; the job time is the
maximum over ranks and the whole-job value counts every rank's FLOPs.
Also the paper's FLOP count (FlashAttention-3, zenmind.me summary §7.1).
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + rank, 50.0 - 7.0 * rank]
    out[rank] = bench.max_over_ranks(local, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [11.0, 50.0]


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.5], 1) == [3.0, 4.5]


def test_job_value_counts_every_rank():
    f = bench.fwd_flops(2, 16, 8192, 128, False) * 4.5
    one = bench.job_tflops(f, 10, 1, 100.0)
    assert bench.job_tflops(f, 10, 2, 100.0) == pytest.approx(2 * one)   # weak scaling: twice the work
    assert bench.job_tflops(f, 10, 2, 200.0) == pytest.approx(one)       # the slowest rank sets the time


def test_flop_formula_of_the_pages():
    # 4 * seqlen^2 * head_dim * heads per batch element, halved when causal
    assert bench.fwd_flops(4, 16, 8448, 128, False) == 4 * 4 * 16 * 8448 ** 2 * 128
    assert bench.fwd_flops(1, 1, 1000, 64, True) == 2 * 1000 ** 2 * 64


@pytest.mark.parametrize("workload", [None, "varlen_t129511_hq32_hkv8_d128_causal",
                                      "decode_fp8_b16_hq32_hkv8_n32768_d128"])
def test_reference_arm_prints_one_contract_line(workload):
    """The reference arm (the oracle on a bounded sample of the workload) runs
    on the host alone and prints one JSON line with the contract's keys."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3"]
    if workload is not None:
        cmd += ["--workload", workload]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["value"] == d["value"] and d["config"]["workload"] == (workload or bench.DEFAULT)
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_clock_samples_are_parsed():
    """nvidia-smi rows (fields of Clocks.Q): median SM clock, max clock, active reasons."""
    text = ("0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "0, 1980, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "0, 2010, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
    r = bench.parse_clock_samples(text)
    assert r == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.parse_clock_samples("") is None
    hot = bench.parse_clock_samples("0, 1500, 2070, 1400, 0x8, Active, Not Active, Active, Not Active\n")
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_samples_outside_the_timed_windows_are_dropped():
    """Timestamped rows: only those inside a (start, end) wall-clock window count."""
    import datetime
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 0)
    row = lambda dt, mhz: (f"{(t0 + datetime.timedelta(seconds=dt)).strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, "
                           f"0, {mhz}, 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    text = row(0.0, 900) + row(1.0, 2070) + row(1.2, 2050) + row(3.0, 1000)
    w = [(t0.timestamp() + 0.9, t0.timestamp() + 1.3)]
    r = bench.parse_clock_samples(text, w)
    assert r["samples"] == 2 and r["sm_mhz"] == 2060.0
    assert bench.parse_clock_samples(text)["samples"] == 4


@pytest.mark.parametrize("workload", [None, "varlen_t129511_hq32_hkv8_d128_causal",
                                      "decode_fp8_b16_hq32_hkv8_n32768_d128"])
def test_reference_arm_other_ranks_exit_quietly(workload):
    """Under a launcher with two ranks, rank 1 of the reference arm does no
    work and prints nothing (rank 0 alone prints the line)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    if workload is not None:
        cmd += ["--workload", workload]
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120, cwd=root, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
