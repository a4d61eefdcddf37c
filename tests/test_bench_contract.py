"""The benchmark's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the keys the benchmark contract asks for, on the same workload
names as the GPU arm.  Runs on the CPU in a second or two per case."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _line(*flags):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", *flags],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("flags,workload", [
    ((), "qwen3next-gdn-verify-b128"),
    (("--kda",), "qwen3next-kda-verify-b128"),
    (("--window", "1"), "qwen3next-gdn-decode-b128"),
    (("--variant", "snapshot", "--batch", "32"), "qwen3next-gdn-snapshot-verify-b32"),
    (("--prefill", "64", "--batch", "2"), "qwen3next-gdn-prefill-b2-n64"),
])
def test_reference_line_follows_the_contract(flags, workload):
    rec = _line(*flags)
    assert KEYS <= rec.keys(), KEYS - rec.keys()
    assert rec["impl"] == "reference" and rec["config"]["workload"] == workload
    assert rec["metric"] in (bench.METRIC, bench.PREFILL_METRIC) and rec["unit"] == "tokens/s"
    assert rec["value"] > 0 and rec["n_gpus"] == 1 and rec["warmup"] == 3
    assert rec["higher_is_better"] is True and rec["scaling"] == "weak"
    assert rec["vs_baseline"] is None and rec["dtype"] == "f64"
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    assert rec["e2e"]["value"] == rec["value"] and rec["e2e"]["unit"] == rec["unit"]


def test_fewer_than_three_warmup_steps_are_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "2"], capture_output=True, text=True,
                       timeout=120, cwd=ROOT)
    assert r.returncode != 0 and "warmup" in r.stderr
