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
    # each step is one request of the workload processed completely: 32 tree tokens per step
    assert d["config"]["tree_tokens_per_step"] == 32
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - 32.0) < 1e-6 * 32.0


def test_oracle_sample_runs_in_a_child_with_the_stated_threads():
    sys.path.insert(0, ROOT)
    import bench
    times = bench.oracle_sample_times(1, 2, 1)
    assert len(times) == 2 and all(t > 0 for t in times)


def test_reference_arm_without_an_oracle_sample_says_so():
    d = _run("--workload", "verify_b8_tree16", "--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference" and "unavailable" in d


def test_clock_sampler_parses_and_cleans_up(tmp_path, monkeypatch):
    """The nvidia-smi sampler of the timed region, against a stand-in
    nvidia-smi that prints two samples (one with sw_power_cap active)."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '0, 2070 MHz, 2070 MHz, 900.00 W, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '0, 1980 MHz, 2070 MHz, 1400.00 W, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ['PATH']}")
    sys.path.insert(0, ROOT)
    import time

    import bench
    c = bench.Clocks(0)
    time.sleep(1.0)
    path = c.path
    got = c.stop()
    assert got == {"sm_mhz": 2025.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}
    assert not os.path.exists(path)
