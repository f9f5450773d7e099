"""Checkpoint and resume: the optimizer's whole state is the momentum M (the
third-level paragraph of "Dion3: Full-Stack Orthogonal Updates" keeps nothing
else; there is no step counter or bias correction) plus, for the lazy step, the
caller-held row_scale.  Five steps, a copy of W, M (and row_scale) to the host,
fresh device tensors and a fresh workspace loaded from that copy, and five more
steps give bit for bit what ten uninterrupted steps give."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from tests._harness import to_dev, to_host

pytestmark = pytest.mark.gpu

SHAPES = [(300, 200, 2, "bf16"), (96, 520, 2, "f32")]


def _grads(t):
    return [[workloads.gaussian((n, m), 0.01, seed=700 + 1000 * t + 10 * gi + b, dtype="bf16")
             for b in range(batch)] for gi, (n, m, batch, _) in enumerate(SHAPES)]


def _fresh(W, M, S):
    Wd = [[to_dev(x, SHAPES[gi][3]) for x in W[gi]] for gi in range(len(SHAPES))]
    Md = [[to_dev(x) for x in M[gi]] for gi in range(len(SHAPES))]
    Sd = [to_dev(s) for s in S]
    return Wd, Md, Sd


def _run(Wd, Md, Sd, t0, t1, hp, lazy):
    sels = [torch.empty((batch, d3.num_selected(hp.f, n)), dtype=torch.int32, device="cuda")
            for (n, m, batch, _) in SHAPES]
    ws = None
    for t in range(t0, t1):
        Gd = [[to_dev(x, "bf16") for x in gs] for gs in _grads(t)]
        groups = [d3.Group(params=Wd[gi], grads=Gd[gi], momentum=Md[gi]) for gi in range(len(SHAPES))]
        if ws is None:
            ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
        if lazy:
            d3.step_lazy(groups, hp, Sd, ws, sel_idx_out=sels)
        else:
            d3.step(groups, hp, ws, sel_idx_out=sels)
    d3.device_status()
    return [s.cpu().numpy() for s in sels]


def _host(Wd, Md, Sd):
    return ([[to_host(x) for x in W] for W in Wd], [[to_host(x) for x in M] for M in Md],
            [to_host(s) for s in Sd])


@pytest.mark.parametrize("lazy", [False, True])
def test_resume_is_bitwise(cuda_lib, lazy):
    hp = d3.HParams(f=0.25, mu=0.95, lr=0.02)
    W0 = [[workloads.gaussian((n, m), 0.02, seed=40 + 10 * gi + b, dtype=pd) for b in range(batch)]
          for gi, (n, m, batch, pd) in enumerate(SHAPES)]
    M0 = [[workloads.gapped_momentum(n, m, seed=60 + 10 * gi + b) for b in range(batch)]
          for gi, (n, m, batch, pd) in enumerate(SHAPES)]
    S0 = [np.ones((batch, n), np.float32) for (n, m, batch, _) in SHAPES]
    # ten uninterrupted steps
    Wd, Md, Sd = _fresh(W0, M0, S0)
    sel_a = _run(Wd, Md, Sd, 0, 10, hp, lazy)
    end_a = _host(Wd, Md, Sd)
    del Wd, Md, Sd
    # five steps, checkpoint to the host, five more on fresh tensors
    Wd, Md, Sd = _fresh(W0, M0, S0)
    _run(Wd, Md, Sd, 0, 5, hp, lazy)
    ck = _host(Wd, Md, Sd)
    del Wd, Md, Sd
    torch.cuda.empty_cache()
    Wd, Md, Sd = _fresh(*ck)
    sel_b = _run(Wd, Md, Sd, 5, 10, hp, lazy)
    end_b = _host(Wd, Md, Sd)
    for a, b in zip(sel_a, sel_b):
        assert np.array_equal(a, b)
    for part_a, part_b in zip(end_a, end_b):
        for a, b in zip(part_a, part_b):
            for x, y in zip(a if isinstance(a, list) else [a], b if isinstance(b, list) else [b]):
                assert np.array_equal(x, y)
    if lazy:
        # the checkpoint carried pending decays (factors != 1)
        assert any((s != 1.0).any() for s in ck[2])
