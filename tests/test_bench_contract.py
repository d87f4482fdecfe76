"""bench.py's JSON line keeps its contract.  The reference arm (the oracle on
the host cores) runs here without a GPU, for the decode, prefill and serving
paths, and its line carries the keys the harness reads."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
        "e2e")


@pytest.mark.parametrize("path", ["decode", "prefill", "serve"])
def test_reference_arm_line(path):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--path", path,
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in KEYS:
        assert k in d, k
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1 and "workload" in d["config"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["warmup"] >= 3


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_reference_arm_line_with_32_token_pages(path):
    """--block-tokens reaches the workload on both paths: the line names the
    page size and keeps its keys."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    wk = "llama1b" if path == "decode" else "prefill8x2k"
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--path", path,
                        "--workload", wk, "--block-tokens", "32", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in KEYS:
        assert k in d, k
    assert d["value"] > 0
    text = json.dumps(d["config"])
    assert "32" in text and ("block_tokens" in text or "32-token" in text), d["config"]
