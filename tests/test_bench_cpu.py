"""The benchmark's output contract, checked without a GPU: the reference arm
(the fp64 oracle timed on the host) prints one JSON line with the contract's
keys; too few warm-up steps are refused; the byte accounting behind the
roofline follows the op definitions."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from backward_normalization_gb300 import synth  # noqa: E402


def _run(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT)


def test_reference_arm_prints_the_contract_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (1, 3, 1)
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert (e["value"], e["unit"], e["h2d_bytes_per_step"], e["d2h_bytes_per_step"]) == \
        (d["value"], d["unit"], 0, 0)


def test_too_few_warmup_steps_are_refused():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "2", timeout=120)
    assert r.returncode != 0
    assert "warmup" in r.stderr


@pytest.mark.parametrize("w", synth.WORKLOADS, ids=[w.name for w in synth.WORKLOADS])
def test_minimal_and_kernel_bytes(w):
    s = {"f32": 4, "f16": 2, "bf16": 2, "f64": 8}[w.dtype]
    mb = bench.min_bytes(w)
    assert mb == {"fwd": 2 * w.E * s, "bwd": 3 * w.E * s}
    kb = bench.kernel_bytes(w, 0, 0)  # two-kernel path: the input is read twice
    assert kb["fwd_stats"] == w.E * s and kb["fwd_apply"] == 2 * w.E * s
    assert kb["bwd_reduce"] == 2 * w.E * s and kb["bwd_dx"] == 3 * w.E * s
    assert bench.esize("f64") == 8
