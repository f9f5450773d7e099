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


@pytest.mark.parametrize("f", [0.25, 1.0])
def test_lazy_matches_oracle_over_steps(cuda_lib, f):
    """dion3_step_lazy against the oracle's (eager) dion3_step over five steps.

    Third-level paragraph of "Dion3: Full-Stack Orthogonal Updates": error
    feedback decays only the selected rows; carrying that decay to the next
    accumulation must not change the method.  After every lazy step: the
    selected rows equal the oracle's (a near tie at the boundary, within fp32
    rounding of the row sums, is handed to the oracle and counted); the momentum
    a caller sees after a flush (dion3_flush_row_scale on copies of M and
    row_scale, so the pending factors still carry into the next step) is
    bit-exact with the oracle's; unselected parameter rows are untouched; W is
    within the step tolerance, and for fp32 parameters the applied update gives
    O within 3e-2 of the oracle's."""
    import math
    from oracle import accumulate, dion3_step, row_l1
    from tests._harness import (O_REL_FRO, SEL_GAP, assert_close_wm, boundary_gap, rel_fro,
                                valid_topk)
    shapes = [(300, 200, 2, "bf16"), (96, 520, 2, "f32"), (130, 64, 1, "f32")]
    hp = d3.HParams(f=f, mu=0.9, lr=0.01)
    f32 = float(np.float32(f))
    lr_eff = float(np.float32(hp.lr / math.sqrt(f32)))
    init = _state(shapes, seed=17)
    Md = [[to_dev(x) for x in Ms] for (Ms, _, _) in init]
    Wd = [[to_dev(x, pd) for x in Ws] for (_, Ws, pd) in init]
    M_o = [[x.copy() for x in Ms] for (Ms, _, _) in init]
    scales = [torch.ones((batch, n), dtype=torch.float32, device="cuda") for (n, m, batch, _) in shapes]
    sels = [torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda")
            for (n, m, batch, _) in shapes]
    ws = None
    near = 0
    for t in range(5):
        grads = [[workloads.gaussian((n, m), 0.01, seed=500 + 1000 * t + 10 * gi + b, dtype="bf16")
                  for b in range(batch)] for gi, (n, m, batch, _) in enumerate(shapes)]
        Gd = [[to_dev(x, "bf16") for x in gs] for gs in grads]
        W_before = [[to_host(x).astype(np.float64) for x in W] for W in Wd]
        groups = [d3.Group(params=Wd[gi], grads=Gd[gi], momentum=Md[gi]) for gi in range(len(shapes))]
        if ws is None:
            ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
        d3.step_lazy(groups, hp, scales, ws, sel_idx_out=sels)
        flushed = []
        for gi in range(len(shapes)):
            Mc = [x.clone() for x in Md[gi]]
            d3.flush_row_scale(Mc, scales[gi].clone())
            flushed.append(Mc)
        d3.device_status()
        for gi, (n, m, batch, pd) in enumerate(shapes):
            idx = sels[gi].cpu().numpy()
            for b in range(batch):
                G = grads[gi][b]
                l1 = row_l1(accumulate(M_o[gi][b], G))
                force = None
                if boundary_gap(l1, idx.shape[1]) < SEL_GAP:
                    assert valid_topk(l1, idx[b], idx.shape[1])
                    force = idx[b]
                    near += 1
                W1, M1, S, O = dion3_step(W_before[gi][b], M_o[gi][b], G, f=f32, mu=hp.mu, lr=hp.lr,
                                          eps=hp.eps, param_dtype=pd, force_selection=force)
                assert np.array_equal(idx[b], S), (t, gi, b)
                assert np.array_equal(to_host(flushed[gi][b]), M1), (t, gi, b)
                Wg = to_host(Wd[gi][b]).astype(np.float64)
                rest = np.setdiff1d(np.arange(n), S)
                assert np.array_equal(Wg[rest], W_before[gi][b][rest])
                assert_close_wm(Wg, W1, f"lazy step {t} group {gi} matrix {b}")
                if pd == "f32":
                    O_gpu = (W_before[gi][b][S] - Wg[S]) / lr_eff
                    assert rel_fro(O_gpu, O) <= O_REL_FRO, (t, gi, b)
                M_o[gi][b] = M1
    assert near <= 2
