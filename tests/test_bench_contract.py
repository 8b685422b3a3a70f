"""bench.py's JSON contract on the host: the reference arm (the oracle timed
on the host cores) prints one line with the contract's keys, its
cpu_baseline and e2e describing the same run, and the GPU arm refuses to run
without a GPU instead of falling back to anything on the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BENCH = os.path.join(ROOT, "bench.py")


def _run(*args, timeout=300):
    return subprocess.run([sys.executable, BENCH, *args], capture_output=True, text=True, timeout=timeout, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    res = _run("--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "b1_s256_h2")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    b = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in b, key
    assert b["impl"] == "reference" and b["n_gpus"] == 1 and b["steps"] == 1 and b["warmup"] == 0
    assert b["higher_is_better"] is True and b["value"] > 0
    assert b["config"]["workload"] == "b1_s256_h2"
    cb = b["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == b["value"] and cb["cores"] >= 1 and cb["sample"] and cb["cpu"]
    assert b["e2e"] == {"value": b["value"], "unit": b["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_refuses_to_run_without_a_gpu():
    res = _run("--steps", "1", "--warmup", "0")
    assert res.returncode != 0
    assert "needs a CUDA GPU" in res.stderr + res.stdout
    assert not [l for l in res.stdout.splitlines() if l.startswith("{")]


@pytest.mark.gpu
def test_gpu_arm_line_on_a_small_workload():
    """One short run of the GPU arm: the contract's keys, the roofline fraction
    as achieved over peak, four launches per step, and the host copies of the
    end-to-end leg sized from the workload's tensors."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    res = _run("--workload", "b1_s256_h2", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    b = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "gpu_launches", "roofline", "clocks",
                "quantise", "cpu_baseline"):
        assert key in b, key
    assert b["steps"] == 5 and b["warmup"] == 3 and b["value"] > 0
    assert b["gpu_launches"] == 4 * 5
    r = b["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    elems = 1 * 256 * 2 * 128
    assert b["e2e"]["h2d_bytes_per_step"] == 3 * elems * 2 and b["e2e"]["d2h_bytes_per_step"] == elems * 2
    assert b["cpu_baseline"]["kind"] == "oracle" and b["cpu_baseline"]["cores"] >= 1
    assert b["quantise"]["algorithmic_bytes"] == 9 * elems
