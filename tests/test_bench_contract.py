"""The benchmark's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the keys the benchmark contract asks for, and the recorded ncu
traffic figures are reported only while the kernel sources they were taken
from are unchanged. Runs without a GPU: neither touches CUDA code."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--workload", "b2h16l8192d64"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "b2h16l8192d64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _bench_module():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_traffic_records_name_their_profile_and_sources():
    """Every recorded DRAM traffic figure points at a committed ncu summary and
    at the kernel sources whose hashes key it."""
    bench = _bench_module()
    assert bench.NCU_TRAFFIC
    for key, rec in bench.NCU_TRAFFIC.items():
        assert rec["bytes"] > 0, key
        assert os.path.isfile(os.path.join(ROOT, rec["profile"])), rec["profile"]
        assert rec["sources"], key
        for rel, digest in rec["sources"].items():
            assert os.path.isfile(os.path.join(ROOT, rel)), rel
            assert len(digest) == 64 and int(digest, 16) >= 0, rel


def test_traffic_is_null_once_a_source_changes(monkeypatch):
    """The figure is reported while every keyed source still has the hash it
    had at the capture, and null as soon as one differs."""
    bench = _bench_module()
    key = next(iter(bench.NCU_TRAFFIC))
    rec = bench.NCU_TRAFFIC[key]
    import hashlib
    current = {rel: hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest()
               for rel in rec["sources"]}
    matching = dict(rec, sources=current)
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, matching)
    assert bench.ncu_traffic(*key) == rec["bytes"]
    rel = next(iter(current))
    stale = dict(rec, sources=dict(current, **{rel: "0" * 64}))
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, stale)
    assert bench.ncu_traffic(*key) is None
    missing = dict(rec, sources=dict(current, **{"no/such/file.cu": "0" * 64}))
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, missing)
    assert bench.ncu_traffic(*key) is None
    assert bench.ncu_traffic("no-such-workload", "bwd", False) is None
