"""dion3_step_normuon against the oracle's NorMuon reading (parity unpinned as
to the pages, which name the per-neuron normalisation but never define it).

* several shape groups, three steps with fresh gradients: indices and momentum
  bit-exact, the unselected rows' state untouched, the selected rows' state v
  within twice O's tolerance (v is a mean of O^2), W within the W tolerance;
* fp32 parameters: the written block's update has Frobenius norm
  lr_eff * rms * sqrt(k m), and every row carries the same scale c once its own
  factor 1 / (sqrt(v) + eps) is taken out (c^2 = (1 - beta2) ms(dW_i) (sqrt(v_i)
  + eps)^2 / v_i on a first step).
"""
import math

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from oracle import accumulate, dion3_step_normuon, row_l1
from tests._harness import O_REL_FRO, assert_close_wm, rel_fro, to_dev, to_host, valid_topk

pytestmark = pytest.mark.gpu

SHAPES = [(300, 200, 3, "bf16"), (96, 520, 2, "f32"), (130, 64, 2, "bf16")]


@pytest.mark.parametrize("f", [0.25, 1.0])
def test_normuon_matches_oracle(cuda_lib, f):
    nm = d3.NormuonParams(beta2=0.9, eps=1e-8, rms=0.2)
    hp = d3.HParams(f=f, mu=0.9, lr=0.01)
    groups, host, vdev, sels = [], [], [], []
    for gi, (n, m, batch, pd) in enumerate(SHAPES):
        Ms = [workloads.gapped_momentum(n, m, seed=40 + 10 * gi + b) for b in range(batch)]
        Ws = [workloads.gaussian((n, m), 0.02, seed=140 + 10 * gi + b, dtype=pd) for b in range(batch)]
        Md = [to_dev(x) for x in Ms]
        Wd = [to_dev(x, pd) for x in Ws]
        v = torch.zeros((batch, n), dtype=torch.float32, device="cuda")
        groups.append((Md, Wd, pd))
        host.append([[to_host(w).astype(np.float64), x.astype(np.float32).copy(), np.zeros(n, np.float32)]
                     for w, x in zip(Wd, Ms)])
        vdev.append(v)
        sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
    ws = None
    for t in range(3):
        cg = []
        for gi, ((Md, Wd, pd), (n, m, batch, _)) in enumerate(zip(groups, SHAPES)):
            Gs = [workloads.gaussian((n, m), 0.01, seed=500 + 100 * t + 10 * gi + b, dtype="bf16")
                  for b in range(batch)]
            cg.append((d3.Group(params=Wd, grads=[to_dev(G, "bf16") for G in Gs], momentum=Md), Gs))
        if ws is None:
            ws = d3.alloc_workspace(d3.workspace_size([c[0] for c in cg], hp))
        v_before = [to_host(v) for v in vdev]
        d3.step_normuon([c[0] for c in cg], hp, nm, vdev, ws, sel_idx_out=sels)
        d3.device_status()
        for gi, ((Md, Wd, pd), (_, Gs)) in enumerate(zip(groups, cg)):
            vg = to_host(vdev[gi])
            S_gpu = sels[gi].cpu().numpy()
            for b in range(len(Md)):
                Wh, Mh, vh = host[gi][b]
                G = np.asarray(Gs[b], dtype=np.float32)
                # the GPU's selection must be a valid top-k of the oracle's l1 (ties
                # within rounding may go either way); the oracle then uses it
                l1 = row_l1(accumulate(Mh, G))
                assert valid_topk(l1, S_gpu[b], S_gpu.shape[1]), (t, gi, b)
                W1, M1, S, O, v1 = dion3_step_normuon(Wh, Mh, G, vh, f=f, mu=hp.mu, lr=hp.lr, beta2=nm.beta2,
                                                      nm_eps=nm.eps, rms=nm.rms, param_dtype=pd,
                                                      force_selection=S_gpu[b])
                assert np.array_equal(to_host(Md[b]), M1), (t, gi, b)
                rest = np.setdiff1d(np.arange(vh.size), S)
                assert np.array_equal(vg[b][rest], v_before[gi][b][rest])
                assert rel_fro(vg[b][S], v1[S]) < 2 * O_REL_FRO, (t, gi, b)
                assert_close_wm(to_host(Wd[b]).astype(np.float64), W1, f"W step {t} group {gi} matrix {b}")
                host[gi][b] = [W1, M1, v1]


@pytest.mark.parametrize("f", [1.0, 0.5])
def test_normuon_update_norm_and_row_factors(cuda_lib, f):
    nm = d3.NormuonParams(beta2=0.95, eps=1e-8, rms=0.2)
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    n, m, batch = 256, 384, 2
    Ms = [workloads.gapped_momentum(n, m, seed=70 + b) for b in range(batch)]
    Ws = [workloads.gaussian((n, m), 0.02, seed=80 + b, dtype="f32") for b in range(batch)]
    Md, Wd = [to_dev(x) for x in Ms], [to_dev(x) for x in Ws]
    G = [to_dev(np.zeros((n, m), np.float32)) for _ in range(batch)]
    v = torch.zeros((batch, n), dtype=torch.float32, device="cuda")
    k = d3.num_selected(f, n)
    sel = torch.empty((batch, k), dtype=torch.int32, device="cuda")
    grp = d3.Group(params=Wd, grads=G, momentum=Md)
    ws = d3.alloc_workspace(d3.workspace_size([grp], hp))
    W0 = [to_host(w).astype(np.float64) for w in Wd]
    d3.step_normuon([grp], hp, nm, [v], ws, sel_idx_out=[sel])
    d3.device_status()
    lr_eff = float(np.float32(hp.lr / math.sqrt(f)))
    vh = to_host(v).astype(np.float64)
    for b in range(batch):
        S = sel[b].cpu().numpy()
        dW = (W0[b] - to_host(Wd[b]).astype(np.float64))[S]
        assert np.linalg.norm(dW) == pytest.approx(lr_eff * nm.rms * math.sqrt(k * m), rel=1e-4)
        vs = vh[b][S]
        c2 = (1.0 - nm.beta2) * np.mean(dW * dW, axis=1) * (np.sqrt(vs) + nm.eps) ** 2 / vs
        assert np.max(np.abs(c2 / np.median(c2) - 1.0)) < 1e-3
