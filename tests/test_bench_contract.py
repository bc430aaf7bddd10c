"""bench.py's host-side contract on CPU: the reference arm's JSON line (the
CPU oracle timed on the host cores), silent non-zero ranks, and the recorded
ncu traffic that is reported only for the sources it was measured on."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run_reference(env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                           "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_json_line():
    r = _run_reference()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "long128k_nq256_h8_d128_kv131072"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_traffic_reported_only_for_measured_sources(monkeypatch):
    import bench
    import qsa_inputs as qi
    w = qi.BY_NAME["long128k_nq256_h8_d128_kv131072"]
    name = next(n for n, r in bench.NCU_TRAFFIC.items() if r["workload"] == w.name)
    rec = bench.NCU_TRAFFIC[name]
    # the record is reported while the kernel's sources are the captured ones
    monkeypatch.setattr(bench, "kernel_source_sha", lambda names: rec["source_sha"])
    assert bench.traffic_for(name, w) == rec["bytes_per_launch"]
    assert bench.traffic_for(name, qi.BY_NAME["mid_nq256_h8_d128_kv32805"]) is None
    assert bench.traffic_for("no_such_kernel", w) is None
    # and not once they have changed
    monkeypatch.setattr(bench, "kernel_source_sha", lambda names: "0" * 16)
    assert bench.traffic_for(name, w) is None


def test_units_and_rates():
    import bench
    import qsa_inputs as qi
    w = qi.BY_NAME["long128k_nq256_h8_d128_kv131072"]
    assert bench.units_per_step(w) == w.nq * w.nb == 256 * 2048
    # whole-job rate: all ranks' units over the slowest rank's milliseconds
    assert bench.aggregate_rate(4, 1000, 2.0) == pytest.approx(4 * 1000 / 2.0e-3)
