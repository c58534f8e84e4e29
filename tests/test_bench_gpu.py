"""bench.py on the GPU: one JSON line that keeps the benchmark contract.

Runs the headline leg and every extra leg with few steps (and the window, sum
and softmax legs on 2^22 floats) in a subprocess, then checks the keys, the
units and that the numbers are consistent with each other.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5",
                          "--warmup", "3", "--cpu-seconds", "1", "--aux-log2n", "22"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_contract_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "clocks", "e2e", "gpu_launches"):
        assert k in line, k
    assert line["unit"] == "TFLOP/s" and line["n_gpus"] == 1 and line["higher_is_better"]
    assert line["steps"] == 5 and line["warmup"] == 3
    assert line["config"]["workload"].startswith("square4096")
    assert line["gpu_launches"] == line["steps"]
    assert line["warm_l2"]["unit"] == "TFLOP/s" and line["warm_l2"]["value"] > 0
    assert line["ms_per_step_min"] <= line["ms_per_step_median"] <= line["ms_per_step_max"]


def test_value_matches_time_and_roofline(line):
    flops = 2 * 4096 ** 3
    assert line["value"] == pytest.approx(flops / (line["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    r = line["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-6)
    assert 0.3 < r["frac"] < 1.1


def test_e2e_and_cpu_baseline(line):
    e = line["e2e"]
    assert e["unit"] == "TFLOP/s"
    assert e["h2d_bytes_per_step"] == 2 * 4096 * 4096 * 4
    assert e["d2h_bytes_per_step"] == 4096 * 4096 * 4
    assert 0 < e["value"] <= line["value"] * 1.05
    assert e["serial_value"] < e["value"]
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0


def test_extra_legs(line):
    t = line["tc3"]
    assert t["unit"] == "TFLOP/s" and t["roofline"]["bound"] == "tensor" and t["value"] > 0
    for leg in ("window5", "sum", "softmax"):
        # 2^22 floats here: written lines may still sit in L2 when a step ends, so the
        # fraction of the copy bandwidth can read above 1; far above means no work.
        r = line[leg]["roofline"]
        assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0.05 < r["frac"] < 1.6, leg
    for lay in ("tn", "nt", "tt"):
        assert line["layouts"][lay]["gemm_f32_ex"]["value"] > 0
        assert line["layouts"][lay]["gemm_f32_tc3_ex"]["value"] > 0
    assert line["contrast"]["gemm_f32_naive"]["value"] < line["value"]


def test_configs_leg_covers_every_configuration(line):
    import bench
    c = line["configs"]
    assert c["peaks"]["unit"] == "TFLOP/s" and c["clocks"]["samples"] >= 0
    for name in bench.CONFIG_WORKLOADS:
        rec = c[name]
        flops = 2 * rec["M"] * rec["N"] * rec["K"]
        for path in ("gemm_f32", "gemm_f32_tc3"):
            r = rec[path]
            assert r["unit"] == "TFLOP/s" and 5 <= r["steps"] <= 50
            assert r["value"] == pytest.approx(flops / (r["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
            assert 0 < r["frac"] < 1.2, (name, path)
    assert c["square4096"]["gemm_f32"]["value"] > c["square4096"]["gemm_f32_naive"]["value"]


def test_tc3_leg_clocks_and_instruction_rate(line):
    r = line["tc3"]["roofline"]
    assert "clocks" in line["tc3"]
    if r["instruction_rate"] is not None:
        assert r["frac_at_instruction_rate"] == pytest.approx(
            r["achieved"] / r["instruction_rate"], rel=1e-6)
        assert 0.1 < r["frac_at_instruction_rate"] < 1.1
    assert set(r["traffic_parts"]) == {"gemm_tc3", "tc3_split_a", "tc3_split_b"}
