"""bench.py's GPU arm prints the one JSON line the benchmark contract asks
for, with the same workload config keys as the reference arm."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_gpu_arm_prints_the_contract_line():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = run_bench("--workload", "decode_T8", "--steps", "50", "--warmup", "3", "--cpu-seconds", "0.5")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "clocks", "gpu_launches"):
        assert key in d, key
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["n_gpus"] == 1 and d["dtype"] == "f32"
    assert d["steps"] == 50 and d["warmup"] == 3 and d["value"] > 0 and d["gpu_launches"] == 50
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["single_thread"]["cores"] == 1
    e = d["e2e"]
    assert e["unit"] == "GB/s" and e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    # the compact sweep of the metric rides on every default line
    sw = d["sweep"]
    assert [r["T"] for r in sw["decode"]] == [1, 2, 4, 8]
    for r in sw["decode"]:
        assert r["H"] == 4096 and r["replays"] >= 21 and r["floor_us"] > 0 and r["us_per_call"] > r["floor_us"]
        # the line rounds each figure to 3 decimals: recomputed from them, within 0.5 %
        want = r["us_per_call"] / (2 * (r["floor_us"] + r["T"] * 106560 / 8e12 * 1e6))
        assert abs(r["vs_2x_floor"] - want) <= 5e-3 * want
    assert [(r["T"], r["H"]) for r in sw["bandwidth"]] == [(512, 8192), (4096, 8192), (8192, 8192), (32768, 8192)]
    assert all(0 < r["frac"] < 1.5 for r in sw["bandwidth"])
    assert sw["bandwidth"][-1]["bitwise_repeat"] is True
    # so do the other outputs and the producer -> finalize pairs
    assert set(d["variants"]) == {"finalize_only", "nvfp4_epilogue", "nvfp4_epilogue_tiled_scales", "expert_rmsnorm"}
    assert all(v["us_per_call"] > 0 for v in d["variants"].values())
    assert {(r["T"], r["busy_cycles"]) for r in d["pdl_pairs"]} >= {(1, 0), (8, 0)}
    ref = run_bench("--impl", "reference", "--workload", "decode_T8", "--steps", "3", "--warmup", "3",
                    "--cpu-seconds", "0.05")
    shared = {k: v for k, v in ref["config"].items() if k != "bytes_per_call"}
    assert all(d["config"][k] == v for k, v in shared.items())
    assert ref["config"]["bytes_per_call"] == d["config"]["bytes_per_call"]
    assert ref["metric"] == d["metric"] and ref["unit"] == d["unit"] and ref["dtype"] == d["dtype"]
