"""Seeded synthetic inputs for the Dion3 optimizer step.

Shared by the tests, ``bench.py`` and the smoke check: it generates momenta,
gradients and parameters with the shapes and value distributions of the
workloads below, and holds none of the method's arithmetic (no accumulation,
selection, normalisation, Newton-Schulz or update).

Workloads (sizes rows x cols; the pages train with ClimbMix data, which is not
available offline, so Gaussian gradients of the right shapes stand in):

* ``single``: one fp32 momentum 256 x 1024 ~ N(0, 1), gradient ~ N(0, 0.01),
  fp32 parameters ~ N(0, 0.02), f = 1, mu = 0.95, lr = 0.02, seed 0.
* ``gapped``: one 1024 x 4096 momentum whose rows have l1 norms on a sorted
  log-uniform [0.1, 10] ladder (times m sqrt(2/pi)), consecutive ratio at least
  1 + 1e-4, rows in random order; bf16 parameters ~ N(0, 0.02); fresh bf16
  gradients ~ N(0, 0.01) per step; f = 1/4, mu = 0.95, 10 steps.
* ``1b`` / ``7b``: the matrix set of a dense transformer (d = 2048, 16 layers /
  d = 4096, 32 layers): attention 4 x d x d, SwiGLU gate/up d x ffn and down
  ffn x d, grouped by shape; bf16 parameters ~ N(0, 0.02), fp32 momentum,
  bf16 gradients ~ N(0, 0.01).
* ``sweep``: fp16 Gaussian X for the Gram-NS sweep, s in {1024 .. 16384},
  L = s x {1, 2, 4, 8}, batch 1 .. 64.

"N(0, 0.01)" is read as standard deviation 0.01.
"""
from __future__ import annotations

import math

import numpy as np

# (rows, cols, matrices per layer) per transformer shape group.
MODEL_SETS = {
    "1b": {"d": 2048, "layers": 16,
           "shapes": [(2048, 2048, 4), (2048, 8192, 2), (8192, 2048, 1)]},
    "7b": {"d": 4096, "layers": 32,
           "shapes": [(4096, 4096, 4), (4096, 11008, 2), (11008, 4096, 1)]},
}


def model_groups(name: str):
    """[(rows, cols, batch)] for a model-shaped matrix set, one entry per shape."""
    spec = MODEL_SETS[name]
    return [(r, c, per * spec["layers"]) for (r, c, per) in spec["shapes"]]


def model_params(name: str) -> int:
    return sum(r * c * b for (r, c, b) in model_groups(name))


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round an array to bf16 with torch's CPU cast and return fp32 values
    (input preparation: the stored inputs are bf16 numbers)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).to(torch.float32).numpy()


def single(seed: int = 0):
    """One fp32 256 x 1024 matrix: M ~ N(0,1), G ~ N(0,0.01), W ~ N(0,0.02)."""
    rng = _rng(seed)
    n, m = 256, 1024
    M = rng.standard_normal((n, m)).astype(np.float32)
    G = (rng.standard_normal((n, m)) * 0.01).astype(np.float32)
    W = (rng.standard_normal((n, m)) * 0.02).astype(np.float32)
    return {"M": M, "G": G, "W": W, "f": 1.0, "mu": 0.95, "lr": 0.02,
            "param_dtype": "f32", "grad_dtype": "f32"}


def ladder(n: int, seed: int, lo: float = 0.1, hi: float = 10.0,
           min_ratio: float = 1.0 + 1e-4) -> np.ndarray:
    """n sorted log-uniform [lo, hi] factors whose consecutive ratio is at least
    ``min_ratio`` (so l1 norms built from them are far apart compared with
    fp32 rounding), in a random order."""
    rng = _rng(seed)
    v = np.sort(np.exp(rng.uniform(math.log(lo), math.log(hi), n)))
    for i in range(1, n):
        v[i] = max(v[i], v[i - 1] * min_ratio)
    return v[rng.permutation(n)]


def gapped_momentum(n: int, m: int, seed: int) -> np.ndarray:
    """Gaussian rows rescaled so their l1 norms follow ``ladder`` times
    m sqrt(2/pi) (the mean l1 of a standard Gaussian row)."""
    rng = _rng(seed + 1)
    X = rng.standard_normal((n, m))
    target = ladder(n, seed) * m * math.sqrt(2.0 / math.pi)
    X *= (target / np.abs(X).sum(axis=1))[:, None]
    return X.astype(np.float32)


def gapped(seed: int = 0, n: int = 1024, m: int = 4096, steps: int = 10):
    """The 1024 x 4096 gapped-ladder workload: M fp32, W bf16 values, one fresh
    bf16 gradient per step (seed + 1000 + step)."""
    M = gapped_momentum(n, m, seed)
    W = to_bf16_values(_rng(seed + 2).standard_normal((n, m)) * 0.02)
    grads = [to_bf16_values(_rng(seed + 1000 + t).standard_normal((n, m)) * 0.01)
             for t in range(steps)]
    return {"M": M, "W": W, "grads": grads, "f": 0.25, "mu": 0.95, "lr": 0.02,
            "param_dtype": "bf16", "grad_dtype": "bf16"}


def gaussian(shape, sigma: float, seed: int, dtype: str = "f32") -> np.ndarray:
    """Seeded Gaussian array with standard deviation ``sigma``; ``dtype`` 'bf16'
    or 'f16' rounds the values to that format (returned as fp32 values)."""
    x = _rng(seed).standard_normal(shape) * sigma
    if dtype == "bf16":
        return to_bf16_values(x)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    return x.astype(np.float32)


def device_gaussian_(t, sigma: float, seed: int):
    """Fill a device tensor in place with seeded N(0, sigma) values (torch's
    Philox generator on the tensor's device); used for the large model-shaped
    sets, which are too big to generate on the host.  Tests that compare a
    matrix of such a set with the oracle copy its inputs to the host before the
    step."""
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed))
    tmp = torch.randn(t.shape, generator=g, device=t.device, dtype=torch.float32)
    t.copy_(tmp.mul_(sigma))
    return t


def device_gapped_before_(M, G, seed: int):
    """Fill the device tensor ``M`` (fp32, n x m) with a previous momentum such
    that the momentum after the next accumulation, M + G, has Gaussian rows whose
    l1 norms follow ``ladder(n, seed)`` times m sqrt(2/pi): the gapped-ladder
    structure (row-norm gaps far above fp32 rounding) on the values that are
    selected from.  The target rows are drawn and rescaled on the device in
    double and ``G`` is taken off them, so the fp32 sum the step forms lies
    within a unit in the last place of the target.  For the model-shaped sets,
    which are too large to build on the host."""
    import torch
    n, m = M.shape
    g = torch.Generator(device=M.device)
    g.manual_seed(int(seed))
    target = torch.randn((n, m), generator=g, device=M.device, dtype=torch.float64)
    l1_target = torch.from_numpy(ladder(n, seed) * m * math.sqrt(2.0 / math.pi)).to(M.device)
    target.mul_((l1_target / target.abs().sum(dim=1))[:, None])
    M.copy_(target.sub_(G.to(torch.float64)))
    return M


SWEEP_S = (1024, 2048, 4096, 8192, 16384)
SWEEP_ASPECT = (1, 2, 4, 8)
SWEEP_BATCH = (1, 4, 16, 64)
