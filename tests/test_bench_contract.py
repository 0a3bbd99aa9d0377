"""bench.py's command-line contract on the host: the reference arm (the oracle
timed on the host cores) prints one JSON line with the required keys, and the
GPU arm fails loudly where there is no GPU (no CPU fallback)."""
import json
import os
import subprocess
import sys

import pytest
import torch

from tests._util import ROOT

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config"}


def _bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    out = _bench("--impl", "reference", "--steps", "2", "--warmup", "1")
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    j = json.loads(lines[0])
    assert REQUIRED <= set(j), REQUIRED - set(j)
    assert j["impl"] == "reference" and j["steps"] == 2 and j["warmup"] == 1 and j["n_gpus"] == 1
    assert j["value"] > 0 and j["ms_per_step"] > 0 and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["cores"] >= 1 and j["cpu_baseline"]["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert j["config"]["workload"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_fails_without_a_gpu():
    out = _bench("--steps", "1", "--warmup", "3", "--e2e-steps", "0", "--no-cpu-baseline")
    assert out.returncode != 0
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
