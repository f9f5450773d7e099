"""dion3_select_rows_noalloc against dion3_select_rows.

The no-workspace variant serves callers that may not allocate device memory
while they step the optimizer; its row-norm scratch is a static array inside
the library.  It must give the same momentum, selected rows and ||M[S]||_F^2
as the workspace entry point, on consecutive calls that reuse (and so see the
leftovers of) that shared scratch.  This file is collected last so that a run
stopping at its first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from tests._harness import to_dev, to_host

pytestmark = pytest.mark.gpu


def _inputs(n, m, batch, seed, gd):
    Ms = [workloads.gapped_momentum(n, m, seed=seed + b) for b in range(batch)]
    Gs = [workloads.gaussian((n, m), 0.01, seed=seed + 100 + b, dtype=gd) for b in range(batch)]
    return Ms, Gs


def _run(fn_noalloc, Ms, Gs, k, gd):
    n, m = Ms[0].shape
    Md = [to_dev(M) for M in Ms]
    Gd = [to_dev(G, gd) for G in Gs]
    idx = torch.full((len(Ms), k), -1, dtype=torch.int32, device="cuda")
    fro2 = torch.full((len(Ms),), -1.0, dtype=torch.float32, device="cuda")
    if fn_noalloc:
        d3.select_rows_noalloc(Md, Gd, k, idx, fro2)
    else:
        ws = d3.alloc_workspace(d3.select_workspace_size(n, m, len(Ms), k))
        d3.select_rows(Md, Gd, k, idx, fro2, ws)
    torch.cuda.synchronize()
    return [to_host(M) for M in Md], idx.cpu().numpy(), fro2.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cuda_lib):
    # First call: a large call filling much of the scratch; second call: a
    # smaller ragged one that reads only what it writes itself.
    cases = [(1024, 4096, 6, 0.25, "bf16", 1), (333, 200, 5, 0.3, "f32", 50)]
    for n, m, batch, f, gd, seed in cases:
        k = d3.num_selected(f, n)
        Ms, Gs = _inputs(n, m, batch, seed, gd)
        M_ref, idx_ref, fro_ref = _run(False, Ms, Gs, k, gd)
        M_got, idx_got, fro_got = _run(True, Ms, Gs, k, gd)
        for b in range(batch):
            assert np.array_equal(M_got[b], M_ref[b])
            assert np.array_equal(idx_got[b], idx_ref[b])
        np.testing.assert_allclose(fro_got, fro_ref, rtol=1e-6, atol=0)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    n, m = 4096, 8
    batch = d3.NOALLOC_MAX_ROWS // n + 1
    M = [torch.zeros((n, m), dtype=torch.float32, device="cuda") for _ in range(1)] * batch
    idx = torch.zeros((batch, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(d3.Dion3Error) as ei:
        d3.select_rows_noalloc(M, None, 1, idx, None)
    assert ei.value.status == d3.ERR_INVALID_ARG
    assert "static scratch" in str(ei.value)
