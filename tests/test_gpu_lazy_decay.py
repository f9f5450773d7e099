"""dion3_step_lazy against dion3_step: over several steps, the selections,
parameters and (flushed) momenta are bit-identical, and the lazy momentum
differs from the eager one exactly on the rows whose decay is pending."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from tests._harness import to_dev, to_host

pytestmark = pytest.mark.gpu


def _state(shapes, seed):
    out = []
    for gi, (n, m, batch, pd) in enumerate(shapes):
        Ms = [workloads.gapped_momentum(n, m, seed=seed + 10 * gi + b) for b in range(batch)]
        Ws = [workloads.gaussian((n, m), 0.02, seed=seed + 100 + 10 * gi + b, dtype=pd) for b in range(batch)]
        out.append((Ms, Ws, pd))
    return out


@pytest.mark.parametrize("f", [0.25, 1.0])
def test_lazy_matches_eager_bitwise(cuda_lib, f):
    shapes = [(300, 200, 3, "bf16"), (96, 520, 2, "f32"), (130, 64, 2, "bf16")]
    init = _state(shapes, seed=5)
    hp = d3.HParams(f=f, mu=0.9, lr=0.01)
    runs = {}
    for lazy in (False, True):
        groups, Md, Wd, sels, scales = [], [], [], [], []
        for (Ms, Ws, pd), (n, m, batch, _) in zip(init, shapes):
            M = [to_dev(x) for x in Ms]
            W = [to_dev(x, pd) for x in Ws]
            Md.append(M)
            Wd.append(W)
            sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
            scales.append(torch.ones((batch, n), dtype=torch.float32, device="cuda"))
        ws = None
        hist = []
        for t in range(4):
            grads = []
            groups = []
            for gi, (n, m, batch, pd) in enumerate(shapes):
                G = [to_dev(workloads.gaussian((n, m), 0.01, seed=1000 * t + 10 * gi + b, dtype="bf16"), "bf16")
                     for b in range(batch)]
                grads.append(G)
                groups.append(d3.Group(params=Wd[gi], grads=G, momentum=Md[gi]))
            if ws is None:
                ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
            if lazy:
                d3.step_lazy(groups, hp, scales, ws, sel_idx_out=sels)
            else:
                d3.step(groups, hp, ws, sel_idx_out=sels)
            d3.device_status()
            hist.append([s.cpu().numpy().copy() for s in sels])
        if lazy:
            # Before the flush the pending rows differ from the eager momenta.
            pending = [to_host(sc) for sc in scales]
            raw = [[to_host(x) for x in M] for M in Md]
            for gi, (n, m, batch, pd) in enumerate(shapes):
                d3.flush_row_scale(Md[gi], scales[gi])
            d3.device_status()
            assert all((to_host(sc) == 1.0).all() for sc in scales)
            runs["pending"], runs["raw"] = pending, raw
        runs[lazy] = (hist, [[to_host(x) for x in M] for M in Md], [[to_host(x) for x in W] for W in Wd])
    (h0, M0, W0), (h1, M1, W1) = runs[False], runs[True]
    for t in range(4):
        for a, b in zip(h0[t], h1[t]):
            assert np.array_equal(a, b)
    for gi in range(len(shapes)):
        for b in range(len(M0[gi])):
            assert np.array_equal(M0[gi][b], M1[gi][b])   # flushed lazy == eager, bitwise
            assert np.array_equal(W0[gi][b], W1[gi][b])
            rows = np.nonzero(runs["pending"][gi][b] != 1.0)[0]
            assert (runs["pending"][gi][b][rows] == np.float32(0.9)).all()
            rest = np.setdiff1d(np.arange(M0[gi][b].shape[0]), rows)
            assert np.array_equal(runs["raw"][gi][b][rest], M0[gi][b][rest])
            # the last step's selected rows are exactly the pending ones
            assert np.array_equal(np.sort(rows), h1[-1][gi][b])


def test_lazy_rejects_missing_scale(cuda_lib):
    hp = d3.HParams(f=0.5)
    M = [torch.zeros((8, 8), device="cuda")]
    W = [torch.zeros((8, 8), device="cuda")]
    G = [torch.zeros((8, 8), device="cuda")]
    g = [d3.Group(params=W, grads=G, momentum=M)]
    ws = d3.alloc_workspace(d3.workspace_size(g, hp))
    with pytest.raises(d3.Dion3Error):
        d3.step_lazy(g, hp, [0], ws)
