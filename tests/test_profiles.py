"""The committed DRAM-traffic record (profiles/traffic.json) that bench.py
reports for the dominant GEMM is consistent with itself, was taken on a small
case (one kernel, a few launches, a few GB on the device), and is used only
while the kernel source is the one it was captured on."""
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


def test_traffic_record_is_a_small_case_capture():
    rec = _record()
    cmd = rec["command"]
    assert "--clock-control none" in cmd
    assert re.search(r"-k regex:\S*gemm", cmd), "one kernel only"
    n = int(re.search(r"-c (\d+)", cmd).group(1))
    assert 1 <= n <= 18, "a few launches only"
    assert "--max-batch" in cmd, "a small case of the bench workload"
    assert rec["device_gb"] <= 8.0


def test_traffic_record_is_consistent():
    rec = _record()
    per_launch = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["launches"]
    assert abs(per_launch - rec["dram_bytes_per_launch_small"]) <= 1.0
    assert rec["dram_bytes_per_launch"] == pytest.approx(rec["dram_bytes_per_launch_small"] * rec["scale"])


def test_bench_uses_the_record_only_for_the_same_source():
    rec = _record()
    with open(os.path.join(ROOT, rec["source"]), "rb") as fh:
        same = hashlib.sha256(fh.read()).hexdigest() == rec["source_sha256"]
    got = _bench().traffic_record("gemm_tcgen05")
    if same:
        assert got is not None and got["dram_bytes_per_launch"] > 0
    else:
        assert got is None
