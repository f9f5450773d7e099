"""The committed profile records match the sources they describe: the DRAM
traffic that bench.py reports for the dominant GEMM (profiles/traffic.json) was
captured on the kernel source as it is now, and is consistent with itself."""
import hashlib
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_matches_current_kernel_source():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)["gemm_tcgen05"]
    with open(os.path.join(ROOT, rec["source"]), "rb") as fh:
        assert hashlib.sha256(fh.read()).hexdigest() == rec["source_sha256"], \
            "kernel changed since the DRAM traffic was captured: re-run the capture in the record's command"
    per_launch = (rec["dram_read_bytes_step"] + rec["dram_write_bytes_step"]) / rec["launches_step"]
    assert abs(per_launch - rec["dram_bytes_per_launch"]) <= 1.0
    assert rec["passes"] == 1 and "--clock-control none" in rec["command"]


def test_bench_reads_the_record():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    rec = bench.traffic_record("gemm_tcgen05")
    assert rec is not None and rec["dram_bytes_per_launch"] > 0
