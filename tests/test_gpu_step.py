"""dion3_step end to end against the oracle.

* single fp32 matrix 256 x 1024, f = 1: indices, momentum (bit-exact), the
  update O recovered from the fp32 parameter change, and W;
* 1024 x 4096 gapped-ladder momentum, f = 1/4, bf16 parameters, 10 steps with
  fresh gradients: indices and the unselected rows bit-exact every step;
* several shape groups with ragged sizes, wide and tall selections.
"""
import math

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from oracle import dion3_step, row_l1, accumulate
from tests._harness import (O_REL_FRO, SEL_GAP, assert_close_wm, boundary_gap, rel_fro, to_dev,
                            to_host, valid_topk)

pytestmark = pytest.mark.gpu


class Mat:
    """One matrix's device state and its oracle twin."""

    def __init__(self, W, M, param_dtype, grad_dtype):
        self.pd, self.gd = param_dtype, grad_dtype
        self.Wd = to_dev(W, param_dtype)
        self.Md = to_dev(M)
        self.W = to_host(self.Wd).astype(np.float64)
        self.M = M.astype(np.float32).copy()


def _step_and_compare(mats, grads, hp, check_o=False):
    """One dion3_step over groups of Mat; the oracle steps each matrix (with the
    GPU's selection where the l1 gap is within rounding).  Returns the number of
    near-tie selections handed to the oracle."""
    groups, sel, gdev = [], [], []
    for ms, gs in zip(mats, grads):
        gd = [to_dev(G, m.gd) for m, G in zip(ms, gs)]
        gdev.append(gd)
        groups.append(d3.Group(params=[m.Wd for m in ms], grads=gd, momentum=[m.Md for m in ms]))
        n = ms[0].M.shape[0]
        k = d3.num_selected(hp.f, n)
        sel.append(torch.full((len(ms), k), -1, dtype=torch.int32, device="cuda"))
    W_before = [[to_host(m.Wd).astype(np.float64) for m in ms] for ms in mats]
    ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
    d3.step(groups, hp, ws, sel_idx_out=sel)
    d3.device_status()
    near = 0
    lr_eff = float(np.float32(hp.lr / math.sqrt(float(np.float32(hp.f)))))
    for gi, (ms, gs) in enumerate(zip(mats, grads)):
        idx = sel[gi].cpu().numpy()
        for b, (m, G) in enumerate(zip(ms, gs)):
            Gv = to_host(to_dev(G, m.gd))  # the gradient values the GPU saw
            l1 = row_l1(accumulate(m.M, Gv))
            k = idx.shape[1]
            force = None
            if boundary_gap(l1, k) < SEL_GAP:
                assert valid_topk(l1, idx[b], k)
                force = idx[b]
                near += 1
            W1, M1, S, O = dion3_step(m.W, m.M, Gv, f=float(np.float32(hp.f)), mu=hp.mu, lr=hp.lr,
                                      eps=hp.eps, param_dtype=m.pd, force_selection=force)
            assert np.array_equal(idx[b], S), (gi, b)
            Mg = to_host(m.Md)
            assert np.array_equal(Mg, M1), (gi, b)  # momentum bit-exact
            Wg = to_host(m.Wd).astype(np.float64)
            rest = np.setdiff1d(np.arange(Wg.shape[0]), S)
            assert np.array_equal(Wg[rest], W_before[gi][b][rest])  # unselected rows untouched
            assert_close_wm(Wg, W1, f"W group {gi} matrix {b}")
            if check_o:
                O_gpu = (W_before[gi][b][S] - Wg[S]) / lr_eff
                assert rel_fro(O_gpu, O) <= O_REL_FRO
            m.W, m.M = Wg, M1
    return near


def test_step_single_fp32_f1(cuda_lib):
    d = workloads.single(seed=0)
    mat = Mat(d["W"], d["M"], "f32", "f32")
    hp = d3.HParams(f=1.0, mu=d["mu"], lr=d["lr"])
    _step_and_compare([[mat]], [[d["G"]]], hp, check_o=True)


def test_step_gapped_ten_steps(cuda_lib):
    d = workloads.gapped(seed=0)
    mat = Mat(d["W"], d["M"], "bf16", "bf16")
    hp = d3.HParams(f=d["f"], mu=d["mu"], lr=d["lr"])
    near = 0
    for t in range(10):
        near += _step_and_compare([[mat]], [[d["grads"][t]]], hp)
    assert near <= 2


@pytest.mark.parametrize("f", [0.3, 1.0])
def test_step_ragged_groups(cuda_lib, f):
    rng = np.random.default_rng(7)
    shapes = [(300, 200, 3, "bf16", "bf16"), (96, 520, 2, "f32", "bf16"), (130, 72, 2, "bf16", "f32")]
    mats, grads = [], []
    for gi, (n, m, batch, pd, gd) in enumerate(shapes):
        ms, gs = [], []
        for b in range(batch):
            M = workloads.gapped_momentum(n, m, seed=100 * gi + b)
            W = workloads.gaussian((n, m), 0.02, seed=1000 + 100 * gi + b, dtype=pd)
            ms.append(Mat(W, M, pd, gd))
            gs.append(workloads.gaussian((n, m), 0.01, seed=2000 + 100 * gi + b, dtype=gd))
        mats.append(ms)
        grads.append(gs)
    hp = d3.HParams(f=f, mu=0.9, lr=0.01)
    for _ in range(2):
        _step_and_compare(mats, grads, hp)


@pytest.mark.parametrize("n,m,f", [(40, 64, 0.01), (64, 1, 0.5), (1, 48, 1.0), (33, 7, 1.0), (8, 8, 1.0)])
def test_step_degenerate_shapes(cuda_lib, n, m, f):
    # k = 1 (one selected row), m = 1 (Gram side 1 on the transpose), n = 1,
    # tiny ragged and square cases.
    M = workloads.gapped_momentum(n, m, seed=n + m) if n > 1 else workloads.gaussian((n, m), 1.0, 5)
    W = workloads.gaussian((n, m), 0.02, seed=6, dtype="bf16")
    G = workloads.gaussian((n, m), 0.01, seed=7, dtype="bf16")
    mat = Mat(W, M, "bf16", "bf16")
    _step_and_compare([[mat]], [[G]], d3.HParams(f=f, mu=0.9, lr=0.01))


def test_step_bf16_ns(cuda_lib):
    # The whole step with bf16 Gram NS: indices and momentum are unaffected
    # (bit-exact), O (recovered from fp32 parameters) within 3e-2.
    d = workloads.single(seed=3)
    mat = Mat(d["W"], d["M"], "f32", "f32")
    hp = d3.HParams(f=0.5, mu=d["mu"], lr=d["lr"], ns_dtype=d3.BF16)
    _step_and_compare([[mat]], [[d["G"]]], hp, check_o=True)
    g = workloads.gapped(seed=1, steps=2)
    mat = Mat(g["W"], g["M"], "bf16", "bf16")
    hp = d3.HParams(f=g["f"], mu=g["mu"], lr=g["lr"], ns_dtype=d3.BF16)
    for t in range(2):
        _step_and_compare([[mat]], [[g["grads"][t]]], hp)
