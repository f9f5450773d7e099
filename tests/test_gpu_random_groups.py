"""Randomised shape groups through the default step, against the oracle.

Each case draws 2-4 shape groups with ragged sizes (rows 8-600, columns 8-700,
some not a multiple of 8, batches 1-5), parameter and gradient dtypes and a
fraction f, and steps them twice in one dion3_step per step (the overlapped
schedule: groups in order, later groups' accumulations pooled into earlier
groups' Newton-Schulz launches where they can be).  Every matrix is checked
against the oracle after each step (selected rows exact, a near tie within fp32
rounding of the row sums handed to the oracle and counted; momentum bit-exact;
unselected parameter rows untouched; W within the step tolerance), and the final
state against the same steps with the overlap off, bit for bit."""
import math

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from oracle import accumulate, dion3_step, row_l1
from tests._harness import SEL_GAP, assert_close_wm, boundary_gap, to_dev, to_host, valid_topk

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(seed)
    ng = int(rng.integers(2, 5))
    groups = []
    for gi in range(ng):
        n = int(rng.integers(8, 601))
        m = int(rng.integers(8, 701))
        if rng.random() < 0.5:
            m = max(8, m // 8 * 8)
        groups.append((n, m, int(rng.integers(1, 6)), str(rng.choice(["bf16", "f32"])),
                       str(rng.choice(["bf16", "f32"]))))
    f = float(rng.choice([0.1, 0.25, 0.3, 0.5, 0.75, 1.0]))
    return groups, f


def _state(groups, seed):
    host = []
    for gi, (n, m, batch, pd, gd) in enumerate(groups):
        mats = []
        for b in range(batch):
            sd = seed * 1000 + 100 * gi + 10 * b
            mats.append({"M": workloads.gapped_momentum(n, m, seed=sd),
                         "W": workloads.gaussian((n, m), 0.02, seed=sd + 1, dtype=pd)})
        host.append(mats)
    return host


def _device(groups, host):
    return [([to_dev(x["W"], pd) for x in mats], [to_dev(x["M"]) for x in mats])
            for (n, m, batch, pd, gd), mats in zip(groups, host)]


def _run(groups, host, f, seed, overlap, check):
    hp = d3.HParams(f=f, mu=0.9, lr=0.01)
    dev = _device(groups, host)
    sels = [torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda")
            for (n, m, batch, pd, gd) in groups]
    oracle_M = [[x["M"].copy() for x in mats] for mats in host]
    f32 = float(np.float32(f))
    near = 0
    d3.set_overlap(overlap)
    try:
        ws = None
        for t in range(2):
            grads = [[workloads.gaussian((n, m), 0.01, seed=seed * 7919 + 1000 * t + 10 * gi + b, dtype=gd)
                      for b in range(batch)] for gi, (n, m, batch, pd, gd) in enumerate(groups)]
            cg = [d3.Group(params=W, grads=[to_dev(x, gd) for x in G], momentum=M)
                  for (W, M), G, (n, m, batch, pd, gd) in zip(dev, grads, groups)]
            W_before = [[to_host(x).astype(np.float64) for x in W] for (W, _) in dev]
            if ws is None:
                ws = d3.alloc_workspace(d3.workspace_size(cg, hp))
            d3.step(cg, hp, ws, sel_idx_out=sels)
            d3.device_status()
            if not check:
                continue
            for gi, (n, m, batch, pd, gd) in enumerate(groups):
                idx = sels[gi].cpu().numpy()
                for b in range(batch):
                    G = grads[gi][b]
                    l1 = row_l1(accumulate(oracle_M[gi][b], G))
                    force = None
                    if boundary_gap(l1, idx.shape[1]) < SEL_GAP:
                        assert valid_topk(l1, idx[b], idx.shape[1])
                        force = idx[b]
                        near += 1
                    W1, M1, S, _ = dion3_step(W_before[gi][b], oracle_M[gi][b], G, f=f32, mu=hp.mu, lr=hp.lr,
                                              eps=hp.eps, param_dtype=pd, force_selection=force)
                    assert np.array_equal(idx[b], S), (seed, t, gi, b)
                    assert np.array_equal(to_host(dev[gi][1][b]), M1), (seed, t, gi, b)
                    Wg = to_host(dev[gi][0][b]).astype(np.float64)
                    rest = np.setdiff1d(np.arange(n), S)
                    assert np.array_equal(Wg[rest], W_before[gi][b][rest])
                    assert_close_wm(Wg, W1, f"seed {seed} step {t} group {gi} matrix {b}")
                    oracle_M[gi][b] = M1
    finally:
        d3.set_overlap(True)
    final = ([[to_host(x) for x in W] for (W, _) in dev], [[to_host(x) for x in M] for (_, M) in dev],
             [s.cpu().numpy() for s in sels])
    return final, near


@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5, 6])
def test_random_groups_match_oracle_and_schedules(cuda_lib, seed):
    groups, f = _case(seed)
    host = _state(groups, seed)
    on, near = _run(groups, host, f, seed, overlap=True, check=True)
    off, _ = _run(groups, host, f, seed, overlap=False, check=False)
    assert near <= 3
    for part_on, part_off in zip(on, off):
        for a, b in zip(part_on, part_off):
            if isinstance(a, list):
                for x, y in zip(a, b):
                    assert np.array_equal(x, y)
            else:
                assert np.array_equal(a, b)
