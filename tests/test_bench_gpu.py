"""bench.py on a GPU, in a short run: the JSON line keeps the benchmark
contract (its keys, units and the arithmetic that ties them together), and
the reference arm prints the same metric on the same workload."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks")


def _run(*args):
    out = subprocess.run([sys.executable, "bench.py", *args], capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_bench_line_keeps_the_contract():
    line = _run("--steps", "6", "--warmup", "3", "--no-extra", "--e2e-steps", "3", "--cpu-seconds", "0.5",
                "--precast-iters", "5", "--reference-iters", "10", "--op-seconds", "0.02", "--evented-steps", "4")
    for k in KEYS:
        assert k in line, k
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, 6, 3)
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    # value and ms_per_step describe the same packs: bytes of one pack per ms
    pack = line["config"]["pack_bytes"]
    assert pack == 302_055_424
    assert line["value"] * line["ms_per_step"] * 1e6 == pytest.approx(pack, rel=1e-9)
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["bytes_per_launch"] == pack
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-12)
    assert r["achieved"] == pytest.approx(line["value"], rel=1e-12)
    assert 0.3 < r["frac"] < 1.3
    e = line["e2e"]
    assert e["unit"] == "GB/s" and e["h2d_bytes_per_step"] == 100_696_064 and e["d2h_bytes_per_step"] == 201_359_360
    assert 0 < e["value"] < line["value"]
    assert line["gpu_launches"] == 6
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert line["clocks"]["sm_mhz"] > 0


def test_reference_arm_matches_the_metric_and_workload():
    ours = _run("--steps", "4", "--warmup", "3", "--no-extra", "--e2e-steps", "0", "--cpu-seconds", "0",
                "--precast-iters", "0", "--reference-iters", "0", "--op-seconds", "0", "--evented-steps", "2")
    ref = _run("--impl", "reference", "--steps", "4", "--warmup", "3")
    assert ref["impl"] == "reference"
    for k in ("metric", "unit", "higher_is_better", "config"):
        assert ref[k] == ours[k], k
    assert ref["e2e"]["h2d_bytes_per_step"] == 0 and ref["cpu_baseline"]["kind"] == "oracle"
