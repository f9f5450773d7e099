"""Pins of the oracle's NorMuon per-neuron normalisation.

The pages never define it (they say only that Dion3 inherits it from NorMuon
and runs it in float32), so these pin the oracle to the definition it states,
not to the pages: per-row running second moment v_i <- beta2 v_i + (1 - beta2)
mean_j O_ij^2, rows divided by sqrt(v_i) + eps, the update rescaled to RMS
`rms` over the written block.  Parity unpinned as to the pages."""
import math

import numpy as np
import pytest

from oracle import dion3_step_normuon, normuon_rows, normuon_update


def _loops_rows(O, v, beta2, eps):
    """The same definition with plain Python loops (a brute-force twin)."""
    d, vn = [], []
    for i, row in enumerate(O.tolist()):
        ms = sum(x * x for x in row) / len(row)
        vv = beta2 * float(v[i]) + (1.0 - beta2) * ms
        vn.append(vv)
        d.append(1.0 / (math.sqrt(vv) + eps))
    return np.array(d), np.array(vn)


def test_rows_match_brute_force_on_a_small_case():
    rng = np.random.default_rng(0)
    O = rng.standard_normal((3, 5))
    v = np.array([0.0, 0.5, 2.0])
    d, vn = normuon_rows(O, v, 0.9, 1e-3)
    d2, vn2 = _loops_rows(O, v, 0.9, 1e-3)
    np.testing.assert_allclose(vn, vn2, rtol=1e-14)
    np.testing.assert_allclose(d, d2, rtol=1e-14)
    # the mean runs over the m = 5 columns of a row, not over the rows
    assert vn[0] == pytest.approx(0.1 * np.mean(O[0] ** 2), rel=1e-14)


def test_without_history_every_row_gets_the_target_rms():
    """beta2 = 0 and eps = 0: each normalised row has mean square 1, so every row
    of the update has mean square rms^2 exactly."""
    rng = np.random.default_rng(1)
    O = rng.standard_normal((7, 11)) * rng.uniform(0.1, 10.0, size=(7, 1))
    d, _ = normuon_rows(O, np.zeros(7), 0.0, 0.0)
    U = normuon_update(O, d, 0.2)
    np.testing.assert_allclose(np.mean(U * U, axis=1), 0.04, rtol=1e-12)


@pytest.mark.parametrize("beta2", [0.0, 0.5, 0.95])
def test_update_frobenius_norm_is_fixed(beta2):
    rng = np.random.default_rng(2)
    O = rng.standard_normal((6, 9))
    v = rng.uniform(0.0, 3.0, size=6)
    d, _ = normuon_rows(O, v, beta2, 1e-8)
    U = normuon_update(O, d, 0.2)
    assert np.linalg.norm(U) == pytest.approx(0.2 * math.sqrt(54), rel=1e-12)
    # the rows keep their directions
    cos = np.sum(U * O, axis=1) / (np.linalg.norm(U, axis=1) * np.linalg.norm(O, axis=1))
    np.testing.assert_allclose(cos, 1.0, rtol=1e-12)


def test_zero_update_and_two_step_history():
    O = np.zeros((2, 4))
    d, vn = normuon_rows(O, np.array([1.0, 2.0]), 0.9, 1e-8)
    np.testing.assert_allclose(vn, [0.9, 1.8])
    assert not np.any(normuon_update(O, d, 0.2))
    rng = np.random.default_rng(3)
    O1, O2 = rng.standard_normal((3, 8)), rng.standard_normal((3, 8))
    _, v1 = normuon_rows(O1, np.zeros(3), 0.95, 1e-8)
    _, v2 = normuon_rows(O2, v1, 0.95, 1e-8)
    want = 0.95 * 0.05 * np.mean(O1 ** 2, axis=1) + 0.05 * np.mean(O2 ** 2, axis=1)
    np.testing.assert_allclose(v2, want, rtol=1e-14)


def test_step_touches_only_the_selected_rows_state():
    rng = np.random.default_rng(4)
    n, m = 8, 12
    W = rng.standard_normal((n, m)) * 0.02
    M = rng.standard_normal((n, m)).astype(np.float32) * np.arange(1, n + 1, dtype=np.float32)[:, None]
    G = np.zeros((n, m), dtype=np.float32)
    v = rng.uniform(0.1, 1.0, size=n).astype(np.float32)
    W1, M1, S, O, v1 = dion3_step_normuon(W, M, G, v, f=0.5, mu=0.9, lr=0.02, param_dtype="f32")
    rest = np.setdiff1d(np.arange(n), S)
    assert np.array_equal(v1[rest], v[rest])
    assert np.array_equal(W1[rest], W[rest])
    assert not np.array_equal(v1[S], v[S])
    # the written block's update has the fixed Frobenius norm (lr_eff rms sqrt(k m)),
    # up to the fp32 rounding of W
    lr_eff = float(np.float32(0.02 / math.sqrt(0.5)))
    dW = W[S] - W1[S]
    assert np.linalg.norm(dW) == pytest.approx(lr_eff * 0.2 * math.sqrt(S.size * m), rel=1e-5)
