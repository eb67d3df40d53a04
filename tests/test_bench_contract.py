"""bench.py's output line: the keys and units the benchmark contract asks for.

The reference arm (the oracle on the host cores) runs here on CPU on the
smallest workload; the GPU arm runs on a GPU at a small size.
"""

import json
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


def _run(args, timeout):
    env = dict(os.environ, PYTHONPATH=str(ROOT))
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def _common(line):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"):
        assert key in line, key
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["data"] == "synthetic" and line["value"] > 0
    assert line["config"]["workload"]
    assert {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(line["e2e"])


def test_reference_arm_line():
    line = _run(["--impl", "reference", "--workload", "tiny-512x1024", "--steps", "1", "--warmup", "1"],
                timeout=600)
    _common(line)
    assert line["impl"] == "reference"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_gpu_arm_line():
    line = _run(["--workload", "gpt2-1.5b-act", "--steps", "200", "--warmup", "5", "--e2e-steps", "5",
                 "--cpu-baseline-seconds", "1"], timeout=900)
    _common(line)
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and 0 < roof["frac"] < 1.2
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert line["gpu_launches"] == 2 * line["steps"]
    assert line["clocks"]["samples"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    for name in ("compress", "decompress_reduce", "reduce_recompress", "compress_fwht", "compress_int8",
                 "decompress_reduce_int8", "decompress_reduce_mma", "emulated_two_shot_allreduce"):
        assert line["kernels"][name]["us"] > 0, name
    assert line["e2e"]["h2d_bytes_per_step"] == 4 * 8192 * 1600 * 2
    # every configuration, each kernel timed alone against the same peak
    import grads_taco_compress_gb300.workloads as W
    assert set(line["by_workload"]) == set(W.WORKLOADS)
    for name, r in line["by_workload"].items():
        for k in ("compress", "decompress_reduce"):
            rec = r[k]
            assert rec["us"] > 0 and abs(rec["frac"] - rec["hbm_gbs"] / roof["peak"]) < 1e-3, (name, k)
    tiny = line["by_workload"]["tiny-512x1024"]
    assert tiny["compress"]["graph_batch"]["us_per_launch"] > 0 and "note" in tiny


def test_profile_hash_ignores_comments():
    """The hash that ties a committed ncu traffic figure to its kernel covers
    code only: a comment edit keeps it, a code edit changes it."""
    sys.path.insert(0, str(ROOT))
    import bench
    a = "int f(int x) {  // scale\n  /* twice */return 2 * x;\n}\n"
    b = "// a new comment\nint f(int x) {\n  return 2 * x;   /* the same code */\n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    for kernel in ("compress", "compress_fwht", "decompress_reduce", "reduce_recompress"):
        assert len(bench.source_hash(kernel)) == 16
