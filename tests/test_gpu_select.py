"""dion3_select_rows (momentum accumulation + l1 top-k) against the oracle:
bit-exact momentum and indices on inputs whose l1 gaps exceed fp32 rounding."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from oracle import accumulate, num_selected, row_l1, row_sumsq, select_rows
from tests._harness import boundary_gap, to_dev, to_host

pytestmark = pytest.mark.gpu


def _select(Ms, Gs, k, grad_dtype):
    n, m = Ms[0].shape
    Md = [to_dev(M) for M in Ms]
    Gd = [to_dev(G, grad_dtype) for G in Gs] if Gs is not None else None
    idx = torch.full((len(Ms), k), -1, dtype=torch.int32, device="cuda")
    fro2 = torch.zeros(len(Ms), dtype=torch.float32, device="cuda")
    ws = d3.alloc_workspace(d3.select_workspace_size(n, m, len(Ms), k))
    d3.select_rows(Md, Gd, k, idx, fro2, ws)
    d3.device_status()
    return [to_host(M) for M in Md], idx.cpu().numpy(), fro2.cpu().numpy()


@pytest.mark.parametrize("n,m,f,gd", [(1024, 4096, 0.25, "bf16"), (777, 1000, 0.3, "f32"),
                                      (300, 36, 0.125, "bf16"), (64, 8, 1.0, "f32")])
def test_select_gapped(cuda_lib, n, m, f, gd):
    batch = 3
    Ms = [workloads.gapped_momentum(n, m, seed=10 + b) for b in range(batch)]
    Gs = [workloads.gaussian((n, m), 0.01, seed=20 + b, dtype=gd) for b in range(batch)]
    k = num_selected(float(np.float32(f)), n)
    Mg, idx, fro2 = _select(Ms, Gs, k, gd)
    for b in range(batch):
        want_M = accumulate(Ms[b], Gs[b])
        assert np.array_equal(Mg[b], want_M)  # bit-exact fp32 sums
        l1 = row_l1(want_M)
        S = select_rows(l1, k)
        if boundary_gap(l1, k) > 1e-5:
            assert np.array_equal(idx[b], S)
        want_f = row_sumsq(want_M)[idx[b]].sum()
        assert abs(fro2[b] - want_f) <= 1e-5 * want_f


def test_select_ties_go_to_lower_index(cuda_lib):
    n, m = 40, 24
    rng = np.random.default_rng(3)
    base = rng.standard_normal((n, m)).astype(np.float32)
    M = base.copy()
    # Rows 5, 17 and 30 are copies of the largest row: exact ties in l1.
    big = base[0] * 50
    for r in (5, 17, 30):
        M[r] = big
    _, idx, _ = _select([M], None, 2, "f32")
    assert list(idx[0]) == [5, 17]
    _, idx, _ = _select([M], None, 3, "f32")
    assert list(idx[0]) == [5, 17, 30]


def test_select_all_zero_rows(cuda_lib):
    M = np.zeros((50, 16), np.float32)
    _, idx, fro2 = _select([M], None, 7, "f32")
    assert list(idx[0]) == list(range(7)) and fro2[0] == 0.0


@pytest.mark.parametrize("k", [1, 100, 333])
def test_select_extreme_k(cuda_lib, k):
    n, m = 333, 64
    M = workloads.gapped_momentum(n, m, seed=4)
    _, idx, _ = _select([M], None, k, "f32")
    assert np.array_equal(idx[0], select_rows(row_l1(M), k))
