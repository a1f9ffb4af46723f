"""The benchmark's final JSON line, built on CPU from made-up timings: it stays under 2 KB,
parses, carries every key the benchmark contract names, and the two arms (the CUDA path and
the oracle's reference arm) print the same ``config``."""

from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches")


def _fake_line(**over):
    kernels = [
        {"name": "rmsnorm", "kernel": "rmsnorm_rows<bf16,vec16,group64,nv4>",
         "bytes": bench.BYTES_RMS, "us": 6.123456789, "GB/s": 5480.123456, "frac": 0.8098765,
         "rows_per_s": 6.7e8, "row": "row",
         "published_context": {"GB/s": 474.0, "note": "x" * 300}},
        {"name": "rope_qk", "kernel": "rope_tiled<bf16,vec16,hpt2>", "bytes": bench.BYTES_RQK,
         "us": 7.5, "GB/s": 5731.0, "frac": 0.847, "rows_per_s": 2.2e10, "row": "head row"},
    ]
    roofline = {"bound": "hbm", "achieved": 5731.0, "peak": 6767.1, "unit": "GB/s",
                "frac": 0.8469, "traffic": 22030000, "kernel": "rope_tiled<bf16,vec16,hpt2>",
                "peak_source": "of measured (hbm_gbs)"}
    cpu = {"value": 3.79, "unit": "GB/s", "cores": 16, "kind": "oracle",
           "sample": "12 whole steps of the workload (fp64 oracle, 16 threads, 10.1 s)",
           "rmsnorm_f32_64x2048_1_thread": {"us": 900.0}}
    e2e = {"value": 325.4, "unit": "GB/s", "h2d_bytes_per_step": 38797312,
           "d2h_bytes_per_step": 37748736, "steps": 200, "ms_per_step": 0.235,
           "schedule": "double-buffered " * 20, "serial": {"value": 188.2, "schedule": "x"},
           "copy_GB/s": 326.0}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_w_max": 800.0,
              "reasons": ["sw_power_cap"], "samples": 11}
    args = dict(value=5621.7, world=1, steps=20, warmup=5, ms_per_step=0.0136, reps=3100,
                M=20, kernels=kernels, roofline=roofline, cpu=cpu, e2e=e2e, clocks=clocks,
                peak=6767.1, detail_path="gpurun_out/bench_detail.json")
    args.update(over)
    return bench.build_line(**args)


def test_line_is_short_parses_and_has_every_key():
    text = bench.line_text(_fake_line())
    assert len(text.encode()) <= 2048
    assert "\n" not in text
    back = json.loads(text)
    for key in REQUIRED:
        assert key in back, key
    assert back["value"] > 0
    assert back["config"]["workload"] == bench.WORKLOAD
    assert back["roofline"]["frac"] > 0 and back["roofline"]["unit"] == "GB/s"
    assert back["cpu_baseline"]["cores"] == 16 and back["cpu_baseline"]["kind"] == "oracle"
    assert back["e2e"]["h2d_bytes_per_step"] > 0 and back["e2e"]["d2h_bytes_per_step"] > 0
    assert back["clocks"]["sm_mhz"] == 2070.0
    assert back["gpu_launches"] == 2 * 20 * 3100
    assert back["timing"]["repeats"] >= 20


def test_line_without_cpu_leg_still_fits():
    back = json.loads(bench.line_text(_fake_line(cpu=None, world=8)))
    assert back["cpu_baseline"] is None and back["n_gpus"] == 8


def test_an_oversized_line_is_refused():
    huge = _fake_line()
    huge["config"] = dict(huge["config"], extra="y" * 4096)
    try:
        bench.line_text(huge)
    except ValueError:
        return
    raise AssertionError("a line over the limit was accepted")


def test_both_arms_print_the_same_config():
    line = _fake_line()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--ref-seconds", "1"],
                       capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0"))
    assert r.returncode == 0, r.stderr
    ref = json.loads(r.stdout.strip().splitlines()[-1])
    assert ref["impl"] == "reference"
    assert ref["config"] == line["config"]
    assert ref["metric"] == line["metric"] and ref["unit"] == line["unit"]
    assert ref["higher_is_better"] == line["higher_is_better"]
    assert len(r.stdout.strip().splitlines()[-1].encode()) <= 2048
