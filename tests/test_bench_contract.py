"""bench.py's output contract, checked on the CPU through its reference (oracle) arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=env)


def test_reference_arm_prints_one_complete_json_line():
    proc = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [l for l in proc.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["gpu_launches"] == 0 and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_on_other_ranks_does_no_work():
    env_rank = dict(os.environ, WORLD_SIZE="2", RANK="1")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                          capture_output=True, text=True, timeout=300, cwd=ROOT, env=env_rank)
    assert proc.returncode == 0, proc.stderr[-2000:]
    assert proc.stdout.strip() == ""


@pytest.mark.parametrize("args", [["--warmup", "2"], ["--path", "nothing"]])
def test_bad_arguments_are_refused(args):
    proc = _run("--impl", "reference", *args, timeout=120)
    assert proc.returncode != 0


def test_both_arms_print_the_same_config():
    """The oracle arm's `config` is the GPU arm's: the same function builds both."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_293_gb300 import workloads
    proc = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert proc.returncode == 0, proc.stderr[-2000:]
    ref = json.loads(proc.stdout.strip().splitlines()[-1])["config"]
    args = argparse.Namespace(workload="tiny", seed=0, l2="alternate")
    ours = bench.workload_config(workloads.make("tiny", seed=0), args, 1)
    assert ref == json.loads(json.dumps(ours))


def test_clock_summary_uses_the_timed_region_then_the_whole_phase():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    row = lambda sm, util, cap: [str(sm), "2070", str(util), "0x0", "Not Active", "Not Active",
                                 "Not Active", "Active" if cap else "Not Active"]
    c.lines = [(1.0, row(600, 0, False)), (2.0, row(2070, 99, False)),
               (3.0, row(2040, 98, True)), (9.0, row(1980, 97, False))]
    c.fast, c.nvml = [], None
    c.windows = [(2.5, 3.5)]                       # one nvidia-smi sample inside
    s = c.summary()
    assert s["sm_mhz"] == 2040 and s["samples"] == 1 and s["sm_max_mhz"] == 2070
    assert s["phase"]["sm_mhz"] == 2040 and s["phase"]["samples"] == 3   # idle sample left out
    assert s["reasons"] == ["sw_power_cap"]
    c.windows = [(4.0, 4.01)]                      # a timed region too short for a sample
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] == s["phase"]["sm_mhz"]
    c.fast = [(4.005, 2055.0, []), (4.008, 2065.0, [])]   # NVML samples inside it
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2060.0 and "NVML" in s["source"]
