"""bench.py's summaries of a launch trace: the GEMM totals and the overlap
summary read the same numbers whether the GEMM launches are traced as one
entry per Newton-Schulz chain or one per role (DION3_TRACE_DETAIL), and the
overlap summary appears exactly when the timed steps carried pooled work."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 7000.0}


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def _entry(ms, flops=0.0, launches=1, nbytes=0.0):
    return {"total_ms": ms, "useful_flops": flops, "launches": launches, "algo_bytes": nbytes}


def _traces(per_role: bool, pooled: bool):
    """Two timed steps and three traced steps without the overlap."""
    if per_role:
        gemm = {"gemm:syrk:1024": _entry(4.0, 2e12, 8), "gemm:sym_square:1024": _entry(10.0, 3e12, 56),
                "gemm:rect:1024": _entry(6.0, 3e12, 8)}
        gemm_alone = {"gemm:syrk:1024": _entry(5.0, 3e12, 12), "gemm:sym_square:1024": _entry(13.5, 4.5e12, 84),
                      "gemm:rect:1024": _entry(7.5, 4.5e12, 12)}
    else:
        gemm = {"gemm_tcgen05": _entry(20.0, 8e12, 72)}
        gemm_alone = {"gemm_tcgen05": _entry(26.0, 12e12, 108)}
    trace = dict(gemm, accum_rownorm=_entry(3.0, nbytes=1e10), scatter_update=_entry(1.0, nbytes=4e9))
    if pooled:
        trace.update(accum_pool=_entry(0.8, nbytes=2e10, launches=2), scatter_pool=_entry(0.2, nbytes=6e9))
    alone = dict(gemm_alone, accum_rownorm=_entry(12.0, nbytes=4.5e10, launches=9),
                 scatter_update=_entry(3.0, nbytes=1.5e10, launches=9))
    return trace, alone


@pytest.mark.parametrize("per_role", [False, True])
def test_gemm_totals_sum_every_gemm_entry(per_role):
    trace, alone = _traces(per_role, pooled=True)
    got = _bench().gemm_totals(trace)
    assert got == {"total_ms": 20.0, "useful_flops": pytest.approx(8e12), "launches": 72}
    assert _bench().gemm_totals(alone)["total_ms"] == 26.0


@pytest.mark.parametrize("per_role", [False, True])
def test_overlap_summary_with_either_trace_naming(per_role):
    trace, alone = _traces(per_role, pooled=True)
    roof, ov = _bench().gemm_alone_and_overlap(trace, 2, alone, 3, PEAKS)
    assert roof["achieved"] == pytest.approx(12e12 / 26e-3 / 1e12)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 1600.0)
    assert roof["frac_burst"] == pytest.approx(roof["achieved"] / 2000.0)
    assert roof["launches_per_step"] == pytest.approx(36.0)
    assert ov["gemm_ms_per_step"] == pytest.approx(10.0)
    assert ov["gemm_ms_per_step_alone"] == pytest.approx(26.0 / 3)
    assert ov["accum_standalone_ms_per_step"] == pytest.approx(1.5)
    assert ov["accum_pool_rest_ms_per_step"] == pytest.approx(0.4)
    assert ov["accum_ms_per_step_alone"] == pytest.approx(4.0)
    assert ov["scatter_standalone_ms_per_step"] == pytest.approx(0.5)
    assert ov["scatter_pool_rest_ms_per_step"] == pytest.approx(0.1)
    assert ov["scatter_ms_per_step_alone"] == pytest.approx(1.0)


def test_no_overlap_summary_without_pooled_work():
    trace, alone = _traces(False, pooled=False)
    roof, ov = _bench().gemm_alone_and_overlap(trace, 2, alone, 3, PEAKS)
    assert ov is None
    assert roof is not None


@pytest.mark.parametrize("per_role", [False, True])
def test_path_fractions_split_gemm_and_memory_work(per_role):
    """The Gram-NS path is every entry with useful FLOPs (its rate against the
    sustained and burst tensor peaks), the select/update path every other
    entry (its algorithmic bytes against the HBM copy bandwidth)."""
    _, alone = _traces(per_role, pooled=False)
    got = _bench().path_fractions(alone, 3, PEAKS)
    tf = 12e12 / 26e-3 / 1e12
    assert got["gram_ns_ms_per_step"] == pytest.approx(26.0 / 3)
    assert got["gram_ns_tflops"] == pytest.approx(tf)
    assert got["gram_ns_frac_sustained"] == pytest.approx(tf / 1600.0)
    assert got["gram_ns_frac_burst"] == pytest.approx(tf / 2000.0)
    gbs = (4.5e10 + 1.5e10) / 15e-3 / 1e9
    assert got["select_update_ms_per_step"] == pytest.approx(5.0)
    assert got["select_update_gbs"] == pytest.approx(gbs)
    assert got["select_update_frac_hbm"] == pytest.approx(gbs / 7000.0)


def test_clock_summary_parses_nvidia_smi_rows():
    """Median SM clock, maximum clock and the throttle reasons seen active, from
    the CSV rows the sampler reads (index, sm, max sm, power, reasons active,
    hw_slowdown, hw_thermal, sw_thermal, sw_power_cap)."""
    rows = ["0, 1500, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1600, 2070, 1395.1, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbled"]
    got = _bench().ClockSampler._summary(rows)
    assert got == {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert _bench().ClockSampler._summary(["", "garbled"]) is None
