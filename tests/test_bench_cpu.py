"""The benchmark's JSON contract, checked on the CPU through its reference
arm (the oracle on the host cores) on the small workload, and its host-side
helpers."""
import json
import os
import subprocess
import sys

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "3",
                        "--warmup", "3", "--reference-seconds", "2"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny" and "model" not in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_threads_keep_four_rows_each():
    assert bench.oracle_threads(16, 32) == 8
    assert bench.oracle_threads(16, 3) == 1
    assert bench.oracle_threads(8, 2048) == 8


def test_oracle_timing_counts_the_gpu_arms_bytes():
    """A whole step through the oracle counts the step's algorithmic K/V bytes
    (each KV head's once, as the GPU arm does), however the rows are dealt
    to threads."""
    from workloads import Workload, make_workload
    for wl in (make_workload("tiny"),
               Workload("gqa_small", 3, 16, 4, 64, 16, "bf16", 64, np.array([5, 40, 130]), seed=3)):
        ref = bench.oracle_state(wl)
        rows = bench.all_rows(wl)
        _, b1 = bench.time_oracle_rows(wl, ref, rows, 1)
        _, b4 = bench.time_oracle_rows(wl, ref, rows, 4)
        assert b1 == b4 == wl.kv_bytes(ref["ctx_lens"])


def test_traffic_keys_of_the_target_configurations():
    from workloads import make_workload
    assert bench.traffic_key(make_workload("long"), False, -1) == "long"
    assert bench.traffic_key(make_workload("long"), False, 512) == "long_p512"
    assert bench.traffic_key(make_workload("prefix", block_size=16), True, -1) == "prefix16_cascade"
    assert bench.traffic_key(make_workload("prefix", block_size=8), False, -1) == "prefix8"
    names = {(w, b, p, c) for w, b, p, c in bench.EXTRA_CONFIGS}
    assert ("gqa8b", None, -1, False) in names and ("long", None, 512, False) in names
    assert {b for w, b, _, c in bench.EXTRA_CONFIGS if w == "prefix" and c} == {8, 16, 32}
