"""Pins for the oracle's Newton-Schulz and Gram Newton-Schulz (CPU only).

Each check compares the oracle with something other than itself: the spectral
closed form through numpy's SVD, the polar factor of a convergent cubic
iteration, and the FLOP figures printed on the pages.
"""
import os

import numpy as np
import pytest

from oracle import (MUON_QUINTIC, gram_newton_schulz, gram_ns_useful_flops,
                    newton_schulz, normalize, standard_ns_dense_flops,
                    standard_ns_useful_flops)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spectral_ns(X, coeffs, steps):
    """Newton-Schulz acts on singular values only: O = U phi^T(Sigma) V^T with
    phi(x) = a x + b x^3 + c x^5 (closed form via the SVD)."""
    a, b, c = coeffs
    U, sig, Vt = np.linalg.svd(X, full_matrices=False)
    for _ in range(steps):
        sig = a * sig + b * sig ** 3 + c * sig ** 5
    return (U * sig) @ Vt


@pytest.mark.parametrize("shape", [(48, 160), (160, 48), (64, 64), (1, 17), (17, 1)])
def test_ns_matches_svd_closed_form(shape):
    rng = np.random.default_rng(11)
    X = normalize(rng.standard_normal(shape), 1e-7)
    got = newton_schulz(X, MUON_QUINTIC, 5)
    want = _spectral_ns(X, MUON_QUINTIC, 5)
    assert got.shape == shape
    assert np.linalg.norm(got - want) <= 1e-12 * max(1.0, np.linalg.norm(want))


def test_ns_detects_swapped_coefficients():
    # The closed form distinguishes coefficient order: a mistake there fails.
    rng = np.random.default_rng(3)
    X = normalize(rng.standard_normal((32, 96)), 1e-7)
    a, b, c = MUON_QUINTIC
    wrong = _spectral_ns(X, (a, c, b), 5)
    assert np.linalg.norm(newton_schulz(X, MUON_QUINTIC, 5) - wrong) > 1e-2


def test_cubic_ns_converges_to_polar_factor():
    # Textbook special case: the cubic map (1.5, -0.5, 0) converges to U V^T for
    # singular values in (0, sqrt(3)).
    rng = np.random.default_rng(5)
    U, _ = np.linalg.qr(rng.standard_normal((12, 12)))
    V, _ = np.linalg.qr(rng.standard_normal((30, 12)))
    sig = np.linspace(0.35, 1.0, 12)
    X = (U * sig) @ V.T
    got = newton_schulz(X, (1.5, -0.5, 0.0), 60)
    assert np.abs(got - U @ V.T).max() < 1e-12


def test_quintic_output_singular_values_cluster_near_one():
    # The quintic map does not converge to 1; it maps well-conditioned inputs
    # into a band around 1.  Gaussian 256 x 1024 input, normalised.
    rng = np.random.default_rng(0)
    X = normalize(rng.standard_normal((256, 1024)), 1e-7)
    sv = np.linalg.svd(newton_schulz(X), compute_uv=False)
    assert sv.min() > 0.68 and sv.max() < 1.2


@pytest.mark.parametrize("shape", [(40, 150), (150, 40), (33, 33)])
@pytest.mark.parametrize("restart", [3, 0, 2, 5])
def test_gram_ns_equals_standard_ns(shape, restart):
    rng = np.random.default_rng(7)
    X = normalize(rng.standard_normal(shape), 1e-7)
    want = newton_schulz(X, MUON_QUINTIC, 5)
    got = gram_newton_schulz(X, MUON_QUINTIC, 5, restart_iter=restart)
    assert got.shape == shape
    assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split()
                vals[key] = float(val)
    return vals


def _gram_flops(s, L, restart):
    log = []
    gram_newton_schulz(np.ones((s, L)) / (s * L), MUON_QUINTIC, 5, restart_iter=restart,
                       op_log=log)
    return gram_ns_useful_flops(log)


def test_flop_model_reproduces_page_savings():
    g = _golden("flop_savings.txt")
    T, alpha = int(g["T"]), g["alpha"]
    s = 16
    L = int(alpha * s)
    gram = _gram_flops(s, L, restart=0)
    sym = standard_ns_useful_flops(s, L, T)
    dense = standard_ns_dense_flops(s, L, T)
    assert round(100 * (1 - gram / sym)) == g["saving_vs_symmetric_percent"]
    assert round(100 * (1 - gram / dense)) == g["saving_vs_dense_percent"]


@pytest.mark.parametrize("restart", [2, 3, 4, 5])
@pytest.mark.parametrize("alpha", [1, 2, 4, 8])
def test_restart_costs_three_alpha_minus_one_n_cubed(restart, alpha):
    g = _golden("flop_savings.txt")
    s = 8
    L = alpha * s
    extra = _gram_flops(s, L, restart) - _gram_flops(s, L, 0)
    assert extra == g["restart_extra_coeff_times_alpha_minus_1"] * (alpha - 1) * s ** 3


def test_gram_ns_flops_closed_form_t5_restart3():
    # 6 s^2 L + 14 s^3 with one restart, 3 s^2 L + 17 s^3 without.
    s, L = 12, 40
    assert _gram_flops(s, L, 3) == 6 * s * s * L + 14 * s ** 3
    assert _gram_flops(s, L, 0) == 3 * s * s * L + 17 * s ** 3
