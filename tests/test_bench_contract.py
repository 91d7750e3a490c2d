"""bench.py's output contract, checked on the CPU through its reference arm
(the fp64 oracle timed on the host cores on a bounded sample of the large
serving step): one JSON line with the contract's keys and types, rank 0 only
under a multi-rank launch, and the recorded DRAM traffic used only while the
profiled kernel sources are unchanged."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--steps", "2", "--warmup", "3", "--ref-step-seconds", "0.2")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k, t in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                 ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                 ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[k], t), k
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["unit"] == "GB/s" and d["data"] == "synthetic" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_prints_on_rank_zero_only():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-step-seconds", "0.1",
               env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_recorded_traffic_follows_the_kernel_sources(monkeypatch):
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    rec = bench.recorded_traffic()
    if rec is None:
        pytest.skip("no traffic record matches the current kernel sources")
    assert rec["bytes_per_launch"] > 0
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0000000000000000")
    assert bench.recorded_traffic() is None
