"""bench.py's reference arm on CPU (no GPU needed): the float64 oracle timed on a bounded
sample, printed as one JSON line with the library arm's metric, unit and config, a
cpu_baseline describing the run and an e2e block with no host<->device bytes. Also with the
regularisers and an aggregation mode, whose config names them in both workloads."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0", *extra],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _check_common(d):
    assert d["impl"] == "reference" and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["unit"] == "valid tokens/s" and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_headline():
    d = _run()
    _check_common(d)
    assert d["metric"].startswith("GRPO loss fwd+bwd valid tokens/s at V=151936 bf16")
    assert d["config"]["vocab"] == 151936 and "loss terms" not in d["config"]["workload"]


@pytest.mark.parametrize("workload", ["qwen_step", "lmhead"])
def test_reference_arm_with_regularisers(workload):
    d = _run("--workload", workload, "--kl", "k3", "--ent-coef", "0.01", "--agg", "seq-mean-token-mean")
    _check_common(d)
    text = d["config"]["terms"] if workload == "lmhead" else d["config"]["workload"]
    assert "KL k3" in text and "entropy bonus coef 0.01" in text and "seq-mean-token-mean" in text
