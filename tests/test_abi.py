"""The C-ABI library loads, exports every symbol of include/dion3.h, and its
host-only paths (validation, sizes, FLOP schedule) behave as documented.

CPU only: no call here launches GPU work.  Calls with valid arguments but fake
device addresses are made only where validation or injected faults return
before any launch.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
from oracle import MUON_QUINTIC, gram_newton_schulz, gram_ns_useful_flops, num_selected

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(d3.LIB_PATH):
        d3.build()
    return d3.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dion3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dion3_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 13
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(d3.EXPORTED) == names


def test_abi_version_and_status_strings(lib):
    assert lib.dion3_abi_version() == d3.ABI_VERSION
    assert lib.dion3_status_string(d3.ERR_WORKSPACE) == b"DION3_ERR_WORKSPACE"
    assert lib.dion3_status_string(99) == b"unknown dion3 status"


@pytest.mark.parametrize("n", [1, 7, 1024, 2048, 4096, 8192, 11008])
@pytest.mark.parametrize("f", [1.0, 0.5, 0.25, 0.125, 0.3, 1e-6])
def test_num_selected_matches_oracle(lib, f, n):
    # The library rounds f to fp32 first; the oracle gets the same fp32 value.
    f32 = float(np.float32(f))
    assert d3.num_selected(f, n) == num_selected(f32, n)


@pytest.mark.parametrize("k,m", [(256, 1024), (1024, 256), (1024, 4096), (2752, 4096), (64, 64)])
@pytest.mark.parametrize("steps,restart", [(5, 3), (5, 0), (5, 2), (5, 5), (3, 3), (1, 0)])
def test_useful_flops_matches_oracle_schedule(lib, k, m, steps, restart):
    log = []
    # The op sequence does not depend on the values or sizes: run a tiny case
    # and relabel its products with this shape's (s, L).
    gram_newton_schulz(np.ones((2, 3)) / 6.0, MUON_QUINTIC, steps, restart_iter=restart, op_log=log)
    s, L = min(k, m), max(k, m)
    log = [(op[0], s, L) if op[0] != "sym" else ("sym", s) for op in log]
    hp = d3.HParams(ns_steps=steps, restart_iter=restart)
    assert d3.useful_flops(k, m, hp) == gram_ns_useful_flops(log)


def test_useful_flops_closed_form(lib):
    s, L = 1024, 4096
    assert d3.useful_flops(s, L, d3.HParams()) == 6 * s * s * L + 14 * s ** 3


def _hp(**kw):
    return d3.HParams(**kw).c_struct()


def test_invalid_hparams_are_rejected(lib):
    out = ctypes.c_size_t(0)
    bad = [dict(restart_iter=1), dict(restart_iter=6), dict(ns_steps=0), dict(eps=-1.0)]
    for kw in bad:
        h = _hp(**kw)
        assert lib.dion3_gram_ns_workspace_size(16, 32, 1, ctypes.byref(h), ctypes.byref(out)) == d3.ERR_INVALID_ARG
        assert lib.dion3_last_error()
    h = _hp(ns_dtype=d3.F32)  # Gram NS runs on 16-bit operands only
    assert lib.dion3_gram_ns_workspace_size(16, 32, 1, ctypes.byref(h), ctypes.byref(out)) == d3.ERR_UNSUPPORTED
    h = _hp(ns_dtype=d3.BF16)
    assert lib.dion3_gram_ns_workspace_size(16, 32, 1, ctypes.byref(h), ctypes.byref(out)) == d3.OK


def _fake_group(rows, cols, batch, base=0x10000, param_dtype=d3.BF16, grad_dtype=d3.BF16, stride=1 << 24):
    arr = ctypes.c_void_p * batch
    P = arr(*[base + i * stride for i in range(batch)])
    G = arr(*[base + (batch + i) * stride for i in range(batch)])
    M = arr(*[base + (2 * batch + i) * stride for i in range(batch)])
    g = d3._Group(rows, cols, batch, param_dtype, grad_dtype,
                  ctypes.cast(P, ctypes.POINTER(ctypes.c_void_p)),
                  ctypes.cast(G, ctypes.POINTER(ctypes.c_void_p)),
                  ctypes.cast(M, ctypes.POINTER(ctypes.c_void_p)))
    return g, (P, G, M)


def test_step_validation_before_any_launch(lib):
    g, keep = _fake_group(64, 48, 2)
    groups = (d3._Group * 1)(g)
    need = ctypes.c_size_t(0)
    hp = _hp(f=0.25)
    assert lib.dion3_workspace_size(groups, 1, ctypes.byref(hp), ctypes.byref(need)) == d3.OK
    assert need.value > 0
    ws = 0x40000000
    # f outside (0, 1]
    for f in (0.0, -0.5, 1.5):
        h = _hp(f=f)
        assert lib.dion3_step(groups, 1, ctypes.byref(h), ws, need.value, None, None) == d3.ERR_INVALID_ARG
    # workspace too small / missing
    assert lib.dion3_step(groups, 1, ctypes.byref(hp), ws, need.value - 1, None, None) == d3.ERR_WORKSPACE
    assert lib.dion3_step(groups, 1, ctypes.byref(hp), None, need.value, None, None) == d3.ERR_WORKSPACE
    # misaligned workspace
    assert lib.dion3_step(groups, 1, ctypes.byref(hp), ws + 16, need.value, None, None) == d3.ERR_INVALID_ARG
    # misaligned tensor pointer
    g2, keep2 = _fake_group(64, 48, 2, base=0x10008)
    groups2 = (d3._Group * 1)(g2)
    assert lib.dion3_step(groups2, 1, ctypes.byref(hp), ws, need.value, None, None) == d3.ERR_INVALID_ARG
    # bad dtype, empty group
    g3, keep3 = _fake_group(64, 48, 2, param_dtype=d3.F16)
    assert lib.dion3_step((d3._Group * 1)(g3), 1, ctypes.byref(hp), ws, need.value, None, None) == d3.ERR_INVALID_ARG
    g4, keep4 = _fake_group(0, 48, 2)
    assert lib.dion3_workspace_size((d3._Group * 1)(g4), 1, ctypes.byref(hp), ctypes.byref(need)) == d3.ERR_INVALID_ARG
    # injected launch failure: valid arguments, no launch, DION3_ERR_CUDA
    assert lib.dion3_workspace_size(groups, 1, ctypes.byref(hp), ctypes.byref(need)) == d3.OK
    os.environ["DION3_INJECT"] = "launch_fail"
    try:
        assert lib.dion3_step(groups, 1, ctypes.byref(hp), ws, need.value, None, None) == d3.ERR_CUDA
        assert b"injected" in lib.dion3_last_error()
    finally:
        del os.environ["DION3_INJECT"]


def test_select_validation(lib):
    M = (ctypes.c_void_p * 1)(0x10000)
    need = ctypes.c_size_t(0)
    assert lib.dion3_select_workspace_size(100, 64, 1, 25, ctypes.byref(need)) == d3.OK
    ws = 0x40000000
    assert lib.dion3_select_rows(100, 64, 1, M, None, d3.F32, 0, 0x2000, 0, ws, need.value, None) == d3.ERR_INVALID_ARG
    assert lib.dion3_select_rows(100, 64, 1, M, None, d3.F32, 101, 0x2000, 0, ws, need.value, None) == d3.ERR_INVALID_ARG
    assert lib.dion3_select_rows(100, 64, 1, None, None, d3.F32, 25, 0x2000, 0, ws, need.value, None) == d3.ERR_INVALID_ARG
    assert lib.dion3_select_rows(100, 64, 1, M, None, d3.F32, 25, 0x2000, 0, ws, 8, None) == d3.ERR_WORKSPACE
    G = (ctypes.c_void_p * 1)(0x20004)
    assert lib.dion3_select_rows(100, 64, 1, M, G, d3.BF16, 25, 0x2000, 0, ws, need.value, None) == d3.ERR_INVALID_ARG


def test_gemm_validation(lib):
    args = dict(mode=d3.GEMM_SYM_LOWER, M=100, N=90, K=64)
    rc = lib.dion3_gemm_f16(args["mode"], 100, 90, 64, 1, 0x10000, 64, 6400, 0x20000, 64, 5760,
                            None, 0, 0, 0x30000, 90, 9000, None, 0, 0, 1.0, 0.0, 0.0, None)
    assert rc == d3.ERR_INVALID_ARG  # symmetric mode needs M == N
    rc = lib.dion3_gemm_f16(d3.GEMM_RECT, 100, 90, 64, 1, 0x10000, 60, 6000, 0x20000, 64, 5760,
                            None, 0, 0, 0x30000, 90, 9000, None, 0, 0, 1.0, 0.0, 0.0, None)
    assert rc == d3.ERR_INVALID_ARG  # lda not a multiple of 8
    rc = lib.dion3_gemm_f16(d3.GEMM_RECT, 100, 90, 64, 1, 0x10008, 64, 6400, 0x20000, 64, 5760,
                            None, 0, 0, 0x30000, 90, 9000, None, 0, 0, 1.0, 0.0, 0.0, None)
    assert rc == d3.ERR_INVALID_ARG  # A not 16-byte aligned
    rc = lib.dion3_gemm_f16(d3.GEMM_RECT, 100, 90, 64, 1, 0x10000, 64, 6400, 0x20000, 64, 5760,
                            None, 0, 0, None, 0, 0, None, 0, 0, 1.0, 0.0, 0.0, None)
    assert rc == d3.ERR_INVALID_ARG  # no output


def test_gemm_half_flag_validation(lib):
    """The half-stored-symmetric flags are checked on the host, before any launch."""
    def call(mode, M, N, K):
        return lib.dion3_gemm_f16(mode, M, N, K, 1, 0x10000, 256, 65536, 0x20000, 256, 65536,
                                  None, 0, 0, 0x30000, 256, 65536, None, 0, 0, 1.0, 0.0, 0.0, None)
    assert call(d3.GEMM_SYM_LOWER | 0x800, 256, 256, 256) == d3.ERR_INVALID_ARG   # unknown flag
    assert call(d3.GEMM_RECT | d3.GEMM_A_TRANS | d3.GEMM_A_HALF, 256, 256, 256) == d3.ERR_INVALID_ARG  # both
    assert call(d3.GEMM_SYM_LOWER | d3.GEMM_A_HALF, 256, 256, 128) == d3.ERR_INVALID_ARG  # A half needs M == K
    assert call(d3.GEMM_RECT | d3.GEMM_B_HALF, 256, 200, 256) == d3.ERR_INVALID_ARG      # B half needs N == K
    assert call(d3.GEMM_RECT | d3.GEMM_OUT_HALF, 256, 256, 256) == d3.ERR_INVALID_ARG    # needs the symmetric mode
    assert b"half" in lib.dion3_last_error() or b"flag" in lib.dion3_last_error()


def test_workspace_grows_with_batch(lib):
    hp = d3.HParams(f=0.25)
    sizes = [d3.gram_ns_workspace_size(256, 1024, b, hp) for b in (1, 2, 8)]
    assert sizes[0] < sizes[1] < sizes[2]
    assert d3.select_workspace_size(1024, 4096, 1, 256) >= 2 * 1024 * 4


@pytest.mark.parametrize("k,m", [(256, 1024), (1024, 256), (2752, 4096), (96, 96)])
def test_variant_flops_match_oracle(lib, k, m):
    from oracle import standard_ns_dense_flops, standard_ns_useful_flops
    hp = d3.HParams(ns_steps=5, restart_iter=3)
    s, L = min(k, m), max(k, m)
    assert d3.ns_useful_flops(d3.NS_STANDARD, k, m, hp) == standard_ns_useful_flops(s, L, 5)
    assert d3.ns_useful_flops(d3.NS_STANDARD_DENSE, k, m, hp) == standard_ns_dense_flops(s, L, 5)
    assert d3.ns_useful_flops(d3.NS_GRAM, k, m, hp) == d3.useful_flops(k, m, hp)
    log = []
    gram_newton_schulz(np.ones((2, 3)) / 6.0, MUON_QUINTIC, 5, restart_iter=3, op_log=log)
    dense = sum(2.0 * s * s * L if op[0] in ("syrk", "rect") else 2.0 * s ** 3 for op in log)
    assert d3.ns_useful_flops(d3.NS_GRAM_DENSE, k, m, hp) == dense
    assert d3.ns_useful_flops(7, k, m, hp) < 0


def test_step_normuon_validation(lib):
    """dion3_step_normuon checks its parameters and state pointers on the host
    before any launch."""
    g, keep = _fake_group(64, 48, 2)
    groups = (d3._Group * 1)(g)
    need = ctypes.c_size_t(0)
    hp = _hp(f=0.25)
    assert lib.dion3_workspace_size(groups, 1, ctypes.byref(hp), ctypes.byref(need)) == d3.OK
    ws = 0x40000000
    v_ok = (ctypes.c_void_p * 1)(0x50000000)
    v_bad = (ctypes.c_void_p * 1)(0x50000002)
    v_null = (ctypes.c_void_p * 1)(None)

    def call(nm, v):
        return lib.dion3_step_normuon(groups, 1, ctypes.byref(hp), nm, v, ws, need.value, None, None)

    good = d3._NormuonParams(0.95, 1e-8, 0.2)
    assert call(None, v_ok) == d3.ERR_INVALID_ARG
    # eps = 0 is refused: a selected row whose O is zero would get d = 1 / 0.
    for bad in ((1.0, 1e-8, 0.2), (-0.1, 1e-8, 0.2), (0.9, -1.0, 0.2), (0.9, 0.0, 0.2), (0.9, 1e-8, 0.0),
                (0.9, 1e-8, float("inf")), (float("nan"), 1e-8, 0.2)):
        assert call(ctypes.byref(d3._NormuonParams(*bad)), v_ok) == d3.ERR_INVALID_ARG, bad
    assert call(ctypes.byref(good), None) == d3.ERR_INVALID_ARG
    assert call(ctypes.byref(good), v_null) == d3.ERR_INVALID_ARG
    assert call(ctypes.byref(good), v_bad) == d3.ERR_INVALID_ARG
    # valid arguments reach the launch stage: the injected failure reports it
    os.environ["DION3_INJECT"] = "launch_fail"
    try:
        assert call(ctypes.byref(good), v_ok) == d3.ERR_CUDA
    finally:
        del os.environ["DION3_INJECT"]


def test_wait_probe_validation(lib):
    """dion3_wait_probe refuses a limit outside [1 us, 1 s] before any launch."""
    for bad in (0, 999, 10**9 + 1, -5):
        assert lib.dion3_wait_probe(0, bad, None) == d3.ERR_INVALID_ARG, bad


def test_set_overlap_toggles(lib):
    """dion3_set_overlap is a host-side switch: it launches nothing."""
    assert lib.dion3_set_overlap(0) == d3.OK
    assert lib.dion3_set_overlap(1) == d3.OK
