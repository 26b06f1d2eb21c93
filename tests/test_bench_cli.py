"""bench.py's reference arm on the CPU: one JSON line with the keys of the
benchmark line, timed on the fp64 oracle (no GPU needed)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _run("--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference"
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "dtype",
              "data", "config", "cpu_baseline", "e2e", "vs_baseline"):
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["unit"] == "tree tokens/s"
    assert d["config"]["workload"] == "longctx_verify_b4_p32k"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the value is the workload's 128 tree tokens per step over the extrapolated step time
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - 128.0) < 1e-6 * 128.0


def test_reference_arm_without_an_oracle_sample_says_so():
    d = _run("--workload", "verify_b8_tree16", "--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference" and "unavailable" in d
