"""Pins for the oracle's selection, rounding and update rule (CPU only)."""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import (accumulate, dion3_step, newton_schulz, normalize, num_selected,
                    round_to_bf16, row_l1, select_rows)


def test_num_selected_is_ceiling_of_f_n():
    assert num_selected(0.25, 1024) == 256
    assert num_selected(0.125, 11008) == 1376
    assert num_selected(0.3, 10) == 3
    assert num_selected(0.31, 10) == 4
    assert num_selected(1.0, 7) == 7
    assert num_selected(1e-9, 7) == 1
    with pytest.raises(ValueError):
        num_selected(0.0, 7)
    with pytest.raises(ValueError):
        num_selected(1.5, 7)


def _dominates(a, b, l1):
    """Row a ranks above row b: larger l1, or equal l1 and lower index."""
    return l1[a] > l1[b] or (l1[a] == l1[b] and a < b)


@pytest.mark.parametrize("seed", range(6))
def test_selection_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = 8
    l1 = rng.integers(0, 4, size=n).astype(np.float64)  # many ties on purpose
    for k in range(1, n + 1):
        valid = [set(c) for c in itertools.combinations(range(n), k)
                 if all(_dominates(a, b, l1) for a in c for b in set(range(n)) - set(c))]
        assert len(valid) == 1
        got = select_rows(l1, k)
        assert list(got) == sorted(valid[0])


def test_round_to_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3e38, 1e-40]])
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_to_bf16(x32.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_to_bf16_brute_force_on_doubles():
    # Nearest bf16 by enumeration of the neighbouring bit patterns, ties to even.
    rng = np.random.default_rng(2)
    xs = rng.standard_normal(3000) * 10.0 ** rng.integers(-5, 5, 3000)
    got = round_to_bf16(xs)
    for x, g in zip(xs, got):
        bits = int(np.array([x], dtype=np.float32).view(np.uint32)[0]) >> 16
        cands = []
        for d in range(-2, 3):
            b = (bits + d) & 0xFFFF
            v = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
            if math.isfinite(v):
                cands.append((abs(v - x), b & 1, v))
        cands.sort()
        best = [c for c in cands if c[0] == cands[0][0]]
        want = min(best, key=lambda c: c[1])[2]  # tie: even mantissa
        assert g == want


def _muon(W, B, grads, lr, mu, eps):
    """Muon in plain double: B <- mu B + G; W <- W - lr NS5(B / (||B|| + eps))."""
    W = W.astype(np.float64).copy()
    B = B.astype(np.float64).copy()
    for G in grads:
        B = mu * B + G
        W = W - lr * newton_schulz(normalize(B, eps))
    return W


def test_full_fraction_reduces_to_muon():
    rng = np.random.default_rng(4)
    n, m, lr, mu = 24, 40, 0.02, 0.95
    W0 = rng.standard_normal((n, m)).astype(np.float32) * 0.02
    M0 = np.zeros((n, m), np.float32)
    grads = [rng.standard_normal((n, m)).astype(np.float32) for _ in range(5)]
    W, M = W0.astype(np.float64), M0
    for G in grads:
        W, M, S, _ = dion3_step(W, M, G, f=1.0, mu=mu, lr=lr, param_dtype="f32",
                                lr_f32=False)
        assert list(S) == list(range(n))
    want = _muon(W0, M0, grads, lr, mu, 1e-7)
    # fp32 storage of W and M is the only difference from plain double.
    assert np.abs(W - want).max() < 1e-6


def test_unselected_rows_untouched_and_lr_scaled():
    rng = np.random.default_rng(8)
    n, m, f, lr = 64, 48, 0.25, 0.02
    W0 = (rng.standard_normal((n, m)) * 0.02).astype(np.float32)
    M0 = rng.standard_normal((n, m)).astype(np.float32)
    G = (rng.standard_normal((n, m)) * 0.01).astype(np.float32)
    W1, M1, S, O = dion3_step(W0, M0, G, f=f, mu=0.95, lr=lr, param_dtype="f32",
                              lr_f32=False)
    assert len(S) == 16
    rest = np.setdiff1d(np.arange(n), S)
    Macc = accumulate(M0, G)
    # Unselected rows: W bitwise unchanged, M holds exactly M + G (not decayed).
    assert np.array_equal(W1[rest], W0[rest].astype(np.float64))
    assert np.array_equal(M1[rest], Macc[rest])
    # Selected rows: M decayed by mu (fp32 product of the fp32 mu).
    assert np.array_equal(M1[S], (np.float32(0.95) * Macc[S]).astype(np.float32))
    # The applied step is (lr / sqrt(f)) O: twice lr O at f = 1/4.
    step = (W0[S].astype(np.float64) - W1[S])
    ratio = np.linalg.norm(step) / np.linalg.norm(O)
    assert abs(ratio - lr / math.sqrt(f)) < 1e-6 * ratio
    # The selected rows are the largest-l1 rows of the accumulated momentum.
    l1 = row_l1(Macc)
    assert l1[S].min() > l1[rest].max()


def test_unselected_rows_keep_accumulating():
    rng = np.random.default_rng(9)
    n, m = 16, 8
    M = np.zeros((n, m), np.float32)
    M[0] = 100.0  # row 0 always dominates
    W = np.zeros((n, m))
    Gs = [(rng.standard_normal((n, m)) * 0.01).astype(np.float32) for _ in range(3)]
    acc = M.copy()
    for G in Gs:
        W, M, S, _ = dion3_step(W, M, G, f=1 / n, mu=0.9, lr=0.1, param_dtype="f32")
        assert list(S) == [0]
        acc = accumulate(acc, G)
    assert np.array_equal(M[1:], acc[1:])


def test_permutation_equivariance():
    rng = np.random.default_rng(10)
    n, m = 32, 20
    W = (rng.standard_normal((n, m)) * 0.02).astype(np.float32)
    M = rng.standard_normal((n, m)).astype(np.float32)
    G = (rng.standard_normal((n, m)) * 0.01).astype(np.float32)
    perm = rng.permutation(n)
    W1, M1, S1, _ = dion3_step(W, M, G, f=0.25, mu=0.95, lr=0.02, param_dtype="bf16")
    W2, M2, S2, _ = dion3_step(W[perm], M[perm], G[perm], f=0.25, mu=0.95, lr=0.02,
                               param_dtype="bf16")
    assert sorted(perm[S2]) == list(S1)
    assert np.array_equal(M2, M1[perm])
    assert np.abs(W2 - W1[perm]).max() <= 1e-12


def test_zero_momentum_gives_zero_update():
    n, m = 8, 12
    W = np.full((n, m), 0.5, np.float32)
    M = np.zeros((n, m), np.float32)
    W1, M1, S, O = dion3_step(W, M, np.zeros_like(M), f=0.5, mu=0.95, lr=0.02,
                              param_dtype="bf16")
    assert list(S) == [0, 1, 2, 3]  # all ties: lowest indices
    assert not O.any() and np.array_equal(W1, W.astype(np.float64))
    assert not M1.any()


def test_tall_selection_runs_ns_on_transpose():
    # k > m: the orthogonalised rows have orthonormal columns (up to the quintic's
    # band), the Muon convention for tall matrices.
    rng = np.random.default_rng(12)
    X = normalize(rng.standard_normal((96, 24)), 1e-7)
    O = newton_schulz(X)
    sv = np.linalg.svd(O, compute_uv=False)
    assert O.shape == (96, 24) and sv.min() > 0.6 and sv.max() < 1.25
