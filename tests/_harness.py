"""Helpers shared by the parity tests: tolerances, selection-gap rule and
host/device conversion.  No method arithmetic lives here."""
from __future__ import annotations

import numpy as np

#: Relative Frobenius error allowed on the orthogonalised update O.
O_REL_FRO = 3e-2
#: |gpu - oracle| <= W_ABS + W_REL |oracle| for updated parameters and momentum.
W_ABS, W_REL = 1e-3, 1e-2
#: Relative l1 gap at the k-th row below which two selections may differ by
#: rounding of the fp32 row sums (above the fp32 tree-sum error
#: (m / 256 + 9) 2^-24 for the sizes used here).
SEL_GAP = 1e-5


def rel_fro(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def assert_close_wm(got, want, what: str):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    bad = np.abs(got - want) > W_ABS + W_REL * np.abs(want)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} entries out of tolerance; "
                           f"worst |diff| {np.abs(got - want).max():.3e}")


def boundary_gap(l1: np.ndarray, k: int) -> float:
    """Relative gap between the k-th and (k+1)-th largest l1 (inf if k == n)."""
    if k >= l1.shape[0]:
        return float("inf")
    v = np.sort(np.asarray(l1, dtype=np.float64))[::-1]
    return float((v[k - 1] - v[k]) / max(v[k - 1], 1e-300))


def valid_topk(l1: np.ndarray, S: np.ndarray, k: int, tol: float = SEL_GAP) -> bool:
    """S is a top-k set of l1 up to a relative tolerance at the boundary."""
    S = np.asarray(S)
    if S.shape != (k,) or len(np.unique(S)) != k or (np.diff(S) <= 0).any():
        return False
    rest = np.setdiff1d(np.arange(l1.shape[0]), S)
    if rest.size == 0:
        return True
    return bool(l1[S].min() >= l1[rest].max() * (1.0 - tol))


def torch_dtype(name: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[name]


def to_dev(x: np.ndarray, dtype: str = "f32"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda").to(torch_dtype(dtype))


def to_host(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy() if t.dtype != torch.float32 else t.detach().cpu().numpy()
