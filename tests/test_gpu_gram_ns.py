"""dion3_gram_ns_batched (fp16 Gram Newton-Schulz on tcgen05) against the
oracle's float64 standard Newton-Schulz of the same (fp16-valued) input."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
from oracle import MUON_QUINTIC, newton_schulz, normalize
from tests._harness import O_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


def _run(X16: np.ndarray, hp: d3.HParams):
    """X16: [batch, k, m] float32 array of fp16-representable values."""
    X = torch.from_numpy(X16).to("cuda").half().contiguous()
    O = torch.full_like(X, float("nan"))
    batch, k, m = X.shape
    ws = d3.alloc_workspace(d3.gram_ns_workspace_size(k, m, batch, hp))
    d3.gram_ns_batched(X, O, hp, ws)
    d3.device_status()
    return O.float().cpu().numpy()


def _inputs(batch, k, m, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((batch, k, m)) * rng.uniform(0.5, 2.0, (batch, 1, 1))
    return X.astype(np.float16).astype(np.float32)


@pytest.mark.parametrize("k,m", [(64, 256), (256, 64), (128, 128), (200, 520), (520, 200),
                                 (256, 1024), (1000, 300), (8, 72), (100, 250), (333, 90)])
@pytest.mark.parametrize("restart", [3, 0])
def test_gram_ns_matches_oracle(cuda_lib, k, m, restart):
    X = _inputs(2, k, m, seed=k * 7 + m)
    hp = d3.HParams(restart_iter=restart)
    O = _run(X, hp)
    assert np.isfinite(O).all()
    for b in range(X.shape[0]):
        want = newton_schulz(normalize(X[b], hp.eps), MUON_QUINTIC, 5)
        err = rel_fro(O[b], want)
        assert err <= O_REL_FRO, (k, m, restart, b, err)


def test_gram_ns_restart_positions(cuda_lib):
    X = _inputs(1, 192, 640, seed=5)
    want = newton_schulz(normalize(X[0], 1e-7), MUON_QUINTIC, 5)
    for rs in (2, 3, 4, 5):
        O = _run(X, d3.HParams(restart_iter=rs))
        assert rel_fro(O[0], want) <= O_REL_FRO, rs


def test_gram_ns_other_schedules(cuda_lib):
    # T = 1 (a single polynomial step) and a textbook cubic map with T = 3.
    X = _inputs(1, 96, 300, seed=9)
    for T, coeffs, rs in ((1, MUON_QUINTIC, 0), (3, (1.5, -0.5, 0.0), 2)):
        hp = d3.HParams(ns_steps=T, restart_iter=rs, coeffs=coeffs)
        O = _run(X, hp)
        want = newton_schulz(normalize(X[0], hp.eps), coeffs, T)
        assert rel_fro(O[0], want) <= O_REL_FRO, (T, coeffs)


def test_gram_ns_zero_input_gives_zero(cuda_lib):
    X = np.zeros((1, 64, 200), np.float32)
    O = _run(X, d3.HParams())
    assert not O.any()


def test_gram_ns_output_singular_values_band(cuda_lib):
    # Workload shape of the single-matrix case: Gaussian 256 x 1024.
    X = _inputs(1, 256, 1024, seed=0)
    O = _run(X, d3.HParams())
    sv = np.linalg.svd(O[0].astype(np.float64), compute_uv=False)
    assert sv.min() > 0.6 and sv.max() < 1.25


def _variant_err(variant, k, m, ns_dtype, seed):
    """Largest relative Frobenius error of a Newton-Schulz variant over a batch
    of two Gaussian k x m matrices (rounded to the 16-bit type), against the
    oracle's float64 standard quintic NS of the same values."""
    tdt = torch.bfloat16 if ns_dtype == d3.BF16 else torch.float16
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((2, k, m)).astype(np.float32)
    hp = d3.HParams(ns_dtype=ns_dtype)
    Xd = torch.from_numpy(X).to("cuda").to(tdt).contiguous()
    O = torch.full_like(Xd, float("nan"))
    ws = d3.alloc_workspace(d3.ns_workspace_size(variant, k, m, 2, hp))
    d3.ns_batched(variant, Xd, O, hp, ws)
    d3.device_status()
    Xv = Xd.float().cpu().numpy().astype(np.float64)
    Og = O.float().cpu().numpy()
    assert np.isfinite(Og).all()
    return max(rel_fro(Og[b], newton_schulz(normalize(Xv[b], hp.eps), MUON_QUINTIC, 5)) for b in range(2))


# Variants and shapes held to the benchmark spec's 3e-2: Gram NS (symmetric
# products) in fp16 everywhere; standard NS (symmetric or dense products) in
# fp16 and bf16 everywhere; dense Gram NS in fp16 and symmetric Gram NS in bf16
# on rectangular shapes.
_MEETS = ([(d3.F16, v, k, m) for v in (0, 2, 3) for (k, m) in ((200, 520), (520, 200), (256, 256), (128, 128))]
          + [(d3.BF16, v, k, m) for v in (2, 3) for (k, m) in ((200, 520), (520, 200), (256, 256), (128, 128))]
          + [(d3.F16, 1, k, m) for (k, m) in ((200, 520), (520, 200), (512, 2048))]
          + [(d3.BF16, 0, k, m) for (k, m) in ((64, 256), (256, 64), (200, 520), (1024, 4096))])


@pytest.mark.parametrize("ns_dtype,variant,k,m", _MEETS)
def test_ns_variants_within_north_star_tolerance(cuda_lib, ns_dtype, variant, k, m):
    err = _variant_err(variant, k, m, ns_dtype, seed=k * 3 + m + variant)
    assert err <= O_REL_FRO, (ns_dtype, variant, k, m, err)


# Variants that do NOT meet the benchmark spec's 3e-2 on square shapes (the
# smallest singular values of a square Gaussian matrix are tiny, and a Gram
# matrix kept in 16 bits loses sigma^2 below the format's precision):
#   * dense Gram NS (every tile, products of two different matrices not
#     mirrored, so their 16-bit asymmetry feeds into later products): fp16
#     2.9e-2 (128 x 128) and 3.4e-2 (256 x 256) measured; bf16 0.06-0.26;
#   * symmetric Gram NS in bf16 (8 significant bits against fp16's 11): 5.8e-2
#     (128 x 128), 5.4e-2 (256 x 256), 3.3e-2 (1024 x 1024) measured.
# These are comparison paths (the Dion3 step runs symmetric Gram NS in fp16, as
# the pages do).  The test holds them to the measured error with a 1.5x margin
# so that a regression still shows; it does not claim the benchmark spec's bound.
_DECLARED = [(d3.F16, 1, 128, 128, 2.9e-2), (d3.F16, 1, 256, 256, 3.4e-2),
             (d3.BF16, 1, 200, 520, 8.7e-2), (d3.BF16, 1, 256, 256, 2.6e-1),
             (d3.BF16, 0, 128, 128, 5.8e-2), (d3.BF16, 0, 256, 256, 5.4e-2),
             (d3.BF16, 0, 1024, 1024, 3.3e-2)]


@pytest.mark.parametrize("ns_dtype,variant,k,m,measured", _DECLARED)
def test_ns_variants_outside_north_star_tolerance_as_declared(cuda_lib, ns_dtype, variant, k, m, measured):
    err = _variant_err(variant, k, m, ns_dtype, seed=k * 3 + m + variant)
    assert err <= 1.5 * measured, (ns_dtype, variant, k, m, err)


def test_gram_ns_s4096_single(cuda_lib):
    """A Gram side of 4096 (the s = 4096, aspect 1 point of the Gram-NS sweep):
    one 4096 x 4096 fp16 Gaussian matrix against the float64 oracle."""
    X = _inputs(1, 4096, 4096, seed=4096)
    O = _run(X, d3.HParams())
    want = newton_schulz(normalize(X[0], 1e-7), MUON_QUINTIC, 5)
    assert rel_fro(O[0], want) <= O_REL_FRO
