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


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("k,m", [(200, 520), (520, 200), (256, 256)])
def test_ns_variants_match_oracle(cuda_lib, variant, k, m):
    # Gram NS (symmetric / dense) and standard NS (symmetric / dense) on the
    # same kernels all compute the oracle's standard quintic NS.
    X = _inputs(2, k, m, seed=variant * 100 + k)
    hp = d3.HParams()
    Xd = torch.from_numpy(X).to("cuda").half().contiguous()
    O = torch.full_like(Xd, float("nan"))
    ws = d3.alloc_workspace(d3.ns_workspace_size(variant, k, m, 2, hp))
    d3.ns_batched(variant, Xd, O, hp, ws)
    d3.device_status()
    O = O.float().cpu().numpy()
    # The product path (variant 0) is held to the step's tolerance.  The other
    # variants are timing references: the dense ones do not mirror products, so
    # the fp16 asymmetry of Z Q and R Z feeds into later products, and standard
    # NS rounds the rectangular iterate five times; they are held to 5e-2.
    tol = O_REL_FRO if variant == 0 else 5e-2
    for b in range(2):
        want = newton_schulz(normalize(X[b], hp.eps), MUON_QUINTIC, 5)
        assert rel_fro(O[b], want) <= tol, (variant, k, m, b)


@pytest.mark.parametrize("k,m", [(64, 256), (256, 64), (200, 520), (1024, 4096), (128, 128)])
def test_gram_ns_bf16_matches_oracle(cuda_lib, k, m):
    # bf16 operands (ns_dtype = BF16): the unit roundoff is 8x that of fp16
    # (2^-8 vs 2^-11), and the error grows accordingly (about 1e-2 here against
    # about 1e-3 for fp16).  Rectangular shapes stay within the step's 3e-2;
    # square ones (the least well-conditioned) are held to 8 x 3e-2.
    rng = np.random.default_rng(k * 3 + m)
    X = rng.standard_normal((2, k, m)).astype(np.float32)
    hp = d3.HParams(ns_dtype=d3.BF16)
    Xd = torch.from_numpy(X).to("cuda").to(torch.bfloat16).contiguous()
    O = torch.full_like(Xd, float("nan"))
    ws = d3.alloc_workspace(d3.gram_ns_workspace_size(k, m, 2, hp))
    d3.gram_ns_batched(Xd, O, hp, ws)
    d3.device_status()
    Xv = Xd.float().cpu().numpy().astype(np.float64)
    Og = O.float().cpu().numpy()
    tol = O_REL_FRO if k != m else 8 * O_REL_FRO
    for b in range(2):
        want = newton_schulz(normalize(Xv[b], hp.eps), MUON_QUINTIC, 5)
        assert rel_fro(Og[b], want) <= tol, (k, m, b, rel_fro(Og[b], want))


def test_gram_ns_s4096_single(cuda_lib):
    """A Gram side of 4096 (the s = 4096, aspect 1 point of the Gram-NS sweep):
    one 4096 x 4096 fp16 Gaussian matrix against the float64 oracle."""
    X = _inputs(1, 4096, 4096, seed=4096)
    O = _run(X, d3.HParams())
    want = newton_schulz(normalize(X[0], 1e-7), MUON_QUINTIC, 5)
    assert rel_fro(O[0], want) <= O_REL_FRO
