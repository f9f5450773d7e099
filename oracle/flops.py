"""Useful-FLOP model of Newton-Schulz variants.

TEST INFRASTRUCTURE ONLY.  Counts follow the first-level paragraph of
"Dion3: Full-Stack Orthogonal Updates" (agihunt summary of the paper): a
symmetric product computes only one triangle, so it is counted as half of the
dense product.  For an s x L input (s <= L):

* a Gram (SYRK) product Y Y^T costs s^2 L useful FLOPs (half of 2 s^2 L);
* a symmetric s x s by s x s product costs s^3 (half of 2 s^3);
* a rectangular Q Y costs 2 s^2 L.

The counts are taken from an op log (``gram_newton_schulz(..., op_log=...)``)
rather than from a closed form, so the schedule the oracle runs is what is
counted.  The tests check them against the page's savings (55 % vs
symmetric-GEMM standard NS, 68 % vs plain NS at T = 5, alpha = 4) and against
the restart cost 3 (alpha - 1) n^3 stated in the page's limitations paragraph.
"""
from __future__ import annotations


def _cost(op) -> float:
    kind = op[0]
    if kind == "syrk":
        _, s, L = op
        return float(s) * s * L
    if kind == "sym":
        _, s = op
        return float(s) ** 3
    if kind == "rect":
        _, s, L = op
        return 2.0 * s * s * L
    raise ValueError(kind)


def gram_ns_useful_flops(op_log) -> float:
    """Sum of useful FLOPs over the op log of one Gram-NS run."""
    return sum(_cost(op) for op in op_log)


def standard_ns_useful_flops(s: int, L: int, steps: int = 5) -> float:
    """Standard NS on X (s x L) with symmetric kernels: per iteration a SYRK
    X X^T (s^2 L), a symmetric square A A (s^3) and a rectangular B X (2 s^2 L)."""
    return steps * (3.0 * s * s * L + float(s) ** 3)


def standard_ns_dense_flops(s: int, L: int, steps: int = 5) -> float:
    """Standard NS with plain (non-symmetric) GEMMs: X X^T (2 s^2 L), A A (2 s^3),
    B X (2 s^2 L) per iteration."""
    return steps * (4.0 * s * s * L + 2.0 * float(s) ** 3)
