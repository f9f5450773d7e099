"""The committed DRAM-traffic record (profiles/traffic.json) that bench.py
reports for the dominant GEMM is consistent with itself, was taken on small
captures (one kernel, a few launches, a few GB on the device each), and is used
only while the kernel source is the one it was captured on."""
import hashlib
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORD = os.path.join(ROOT, "profiles", "traffic.json")


def _bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def _record():
    if not os.path.exists(RECORD):
        pytest.skip("no traffic record committed")
    with open(RECORD) as fh:
        return json.load(fh)["gemm_tcgen05"]


def test_traffic_captures_are_small():
    rec = _record()
    assert rec["captures"]
    for cap in rec["captures"]:
        cmd = cap["command"]
        assert "--clock-control none" in cmd
        assert re.search(r"-k regex:\S*gemm", cmd), "one kernel only"
        n = int(re.search(r"-c (\d+)", cmd).group(1))
        assert 1 <= n <= 18 and cap["launches"] == n, "a few launches only"
        assert "--sweep-points" in cmd or "--max-batch" in cmd, "a small case, not the whole set"
        assert cap["device_gb"] <= 8.0
        assert "--set full" not in cmd and "--section" not in cmd


def test_traffic_record_is_consistent():
    rec = _record()
    caps = rec["captures"]
    assert rec["launches"] == sum(c["launches"] for c in caps)
    assert rec["dram_read_bytes"] == sum(c["dram_read_bytes"] for c in caps)
    assert rec["dram_write_bytes"] == sum(c["dram_write_bytes"] for c in caps)
    per_launch = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["launches"]
    assert rec["dram_bytes_per_launch"] == pytest.approx(per_launch)


def test_bench_uses_the_record_only_for_the_same_source():
    rec = _record()
    with open(os.path.join(ROOT, rec["source"]), "rb") as fh:
        same = hashlib.sha256(fh.read()).hexdigest() == rec["source_sha256"]
    got = _bench().traffic_record("gemm_tcgen05")
    if same:
        assert got is not None and got["dram_bytes_per_launch"] > 0
    else:
        assert got is None


def test_record_is_used_only_for_its_own_workload():
    """The record names the workload its captures were taken on; bench.py
    attaches it to that workload's line only (another workload, f, operand
    type or a capped batch gets no traffic figure)."""
    rec = _record()
    wl = rec["workload"]
    bench = _bench()
    with open(os.path.join(ROOT, rec["source"]), "rb") as fh:
        same = hashlib.sha256(fh.read()).hexdigest() == rec["source_sha256"]
    if same:
        assert bench.traffic_record("gemm_tcgen05", dict(wl)) is not None
    for key, other in (("workload", "gapped"), ("f", 0.125), ("ns_dtype", "bf16"), ("max_batch", 4)):
        assert bench.traffic_record("gemm_tcgen05", dict(wl, **{key: other})) is None
