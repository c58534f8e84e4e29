"""bench.py host logic on CPU: rank aggregation over two gloo processes, clock parsing,
the FFMA peak, and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # Rank r takes 1 + r ms for 10 FLOP: max time and summed FLOPs are the job's numbers.
    ms, flops = bench.reduce_over_ranks(dist, 1.0 + rank, 10.0)
    bench.barrier(dist)
    q.put((rank, ms, flops))
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.0, 20.0), (1, 2.0, 20.0)]


def test_single_rank_reduce_is_identity():
    assert bench.reduce_over_ranks(None, 3.5, 7.0) == (3.5, 7.0)


def test_ffma_peak_formula():
    peak, how = bench.ffma_peak_tflops(152, {"sm_max_mhz": 2070.0})
    assert abs(peak - 152 * 128 * 2 * 2070e6 / 1e12) < 1e-9
    assert "152 SMs" in how
    fallback, how = bench.ffma_peak_tflops(152, {})
    assert fallback == peak and "fallback" in how


def test_clock_sampler_parses_nvidia_smi_lines():
    s = bench.ClockSampler(None)
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout: 0})()
    s.lines = ["1965, 2070, 850.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "2070, 2070, 900.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    out = s.stop()
    assert out["samples"] == 2
    assert out["sm_mhz"] == (1965 + 2070) / 2
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "square256", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "square256", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0
    assert res.stdout.strip() == ""
