"""The benchmark's JSON line contract, checked on CPU.

The GPU arm's measurements are replaced by fixed fakes, so only the assembly
of the line is exercised: every key the line promises is present with the
right type.  The reference arm (the oracle on the host cores) runs for real on
a short budget.
"""
import json
import os
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
             "cpu_baseline", "e2e"}


def test_gpu_arm_line_assembly(monkeypatch, capsys):
    import torch
    import bench
    monkeypatch.setattr(torch.cuda, "set_device", lambda *a, **k: None)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    monkeypatch.setattr(torch.cuda, "current_device", lambda *a, **k: 0)
    monkeypatch.setitem(sys.modules, "dequant_gemv_moe_gb300",
                        types.ModuleType("dequant_gemv_moe_gb300"))
    lay = {"ms_per_step": 0.034, "weight_bytes": bench.LAYER_WEIGHT_BYTES, "act_bytes": 225280,
           "value": 3600.0, "kern_ms": 0.0085, "kern_src": "events", "serialised_launch_ms": 0.015,
           "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3},
           "launches": 40, "n_linears": 4,
           "timing": {"repetitions": 7, "ms_per_step_median": 0.034, "ms_per_step_p10": 0.033,
                      "ms_per_step_p90": 0.036},
           "e2e": {"value": 2000.0, "unit": "GB/s", "h2d_bytes_per_step": 53248,
                   "d2h_bytes_per_step": 172032}}
    monkeypatch.setattr(bench, "bench_layer", lambda *a, **k: dict(lay))
    monkeypatch.setattr(bench, "bench_gemv_70b",
                        lambda *a, **k: {"shape": "28672x8192", "us_median": 30.0, "us_p10": 29.0,
                                         "us_p90": 31.0, "us_back_to_back": 24.0,
                                         "us_back_to_back_p10": 23.5, "us_back_to_back_p90": 24.5,
                                         "weight_GBps": 4000.0, "weight_GBps_back_to_back": 5500.0})
    monkeypatch.setattr(bench, "bench_gemv_70b_formats",
                        lambda *a, **k: {"f": {"weight_GBps": 1.0, "weight_GBps_back_to_back": 2.0}})
    monkeypatch.setattr(bench, "bench_dequant",
                        lambda *a, **k: {"q4_k_28672x8192": {"us": 200.0, "bytes": 1,
                                                             "GBps": 5000.0}})
    monkeypatch.setattr(bench, "bench_moe", lambda *a, **k: {"GBps": 100.0, "tokens_per_s": 1.0,
                                                           "expert_tflops": 50.0})
    monkeypatch.setattr(bench, "bench_moe_streamed", lambda *a, **k: {})
    monkeypatch.setattr(bench, "oracle_sample_isolated",
                        lambda *a, **k: {"value": 0.8, "unit": "GB/s", "cores": 8, "kind": "oracle",
                                         "sample": "rows"})
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "10", "--warmup", "3"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.run_ours(bench.parse())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert BASE_KEYS <= set(line)
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["warmup"] == 3
    assert line["value"] == pytest.approx(bench.LAYER_WEIGHT_BYTES / 0.034e-3 / 1e9, rel=1e-3)
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None and line["data"] == "synthetic"
    assert "workload" in line["config"]
    rf = line["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(rf)
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    cb = line["cpu_baseline"]
    assert {"value", "unit", "cores", "kind", "sample"} <= set(cb) and cb["kind"] == "oracle"
    assert {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(line["e2e"])
    assert line["gpu_launches"] == 40 * 7
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])
    # the workload config carries no measurement; the 70B gate GEMV sits in the roofline
    assert "frac_of_hbm" not in line["config"]
    ns = rf["gemv_70b_gate_b1"]
    assert ns["bar"] == 0.8 and ns["meets_bar_back_to_back"] is True
    assert ns["frac_back_to_back"] == pytest.approx(5500.0 / rf["peak"], rel=1e-3)
    assert line["timing"]["repetitions"] == 7


def test_cpu_baseline_in_its_own_process():
    import bench
    r = bench.oracle_sample_isolated(budget_s=0.5, threads=2)
    assert r["kind"] == "oracle" and r["cores"] == 2 and r["value"] > 0
    assert "whole passes" in r["sample"]


def test_reference_arm_runs_the_oracle():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert BASE_KEYS <= set(line)
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # both arms describe the same workload
    import bench
    assert line["config"]["workload"] == bench.layer_config(1)["workload"]
