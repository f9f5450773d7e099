"""Dion3 optimizer step: plain, slow, float64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).  numpy, float64, no
blocking, no fusion, no reordering beyond what the method states.

Sources, by page title and passage:

* "Dion3: Full-Stack Orthogonal Updates" (agihunt summary of the paper),
  paragraph on the *first level* (algorithm): Newton-Schulz normally iterates on
  the large input X; Dion3 iterates on the small symmetric Gram matrix X X^T and
  multiplies back by X at the end; the output equals standard Newton-Schulz; a
  restart at iteration 3; float16 on the GPU.
* same page, paragraph on the *third level* (row selection): pick
  k = ceil(f n) rows of the momentum by l1 norm, orthogonalise only that
  sub-matrix, update only the matching weight rows, decay only the selected
  momentum rows by a factor mu (error feedback), leave the other rows as they
  are; f = 1 gives back Muon; learning rate scaled as eta ~ 1/sqrt(f).
* "Dion3 Cuts Muon Optimizer Time by Up to 6x ...", section "Dion3's fastest
  path is a combined systems stack": error feedback carries what one update
  leaves out into later steps; a full-fraction configuration is Muon in exact
  arithmetic.

Readings taken where the pages are silent (each is also listed in the design
notes of the repository):

* Momentum form (error feedback): M <- M + G on every row, select on the
  accumulated M, orthogonalise the undecayed selected rows, then decay only the
  selected rows by mu.  At f = 1 this is Muon's B_t = mu B_{t-1} + G_t.
* Selection: largest l1 first, ties to the lower row index, S sorted ascending;
  k = ceil(f n) evaluated in double, clamped to [1, n].
* Normalisation before Newton-Schulz: X / (||X||_F + eps).
* Orientation: when k > m, Newton-Schulz runs on X^T (the Gram matrix is formed
  on the short side) and the result is transposed back; same polar factor.
* Quintic coefficients (a, b, c) = (3.4445, -4.7750, 2.0315) for all T = 5
  iterations; the pages print none.
* lr_eff = lr / sqrt(f) (proportionality constant 1: parity unpinned as to the
  constant, since the pages give only the proportionality); no weight decay.
* NorMuon per-neuron normalisation is mentioned but never defined on the pages.
  ``dion3_step`` leaves it out.  ``dion3_step_normuon`` adds it as a reading
  taken from the NorMuon method itself (PARITY UNPINNED as to the pages: they
  only say the normalisation is NorMuon's and runs in float32).  The reading's
  definition is in ``normuon_rows`` / ``normuon_update``; its CPU tests pin the
  code to that definition (closed forms and invariants), not to the pages.
* Rounding: M is stored in fp32 (each + and x computed exactly in double, then
  rounded once to fp32 round-to-nearest-even, which equals an fp32 operation);
  the parameter update is computed in double and rounded once to the parameter
  dtype (fp32 or bf16, RNE).
"""
from __future__ import annotations

import math

import numpy as np

#: Muon's quintic Newton-Schulz coefficients (a, b, c).
MUON_QUINTIC = (3.4445, -4.7750, 2.0315)


# ----------------------------------------------------------------------------
# Step (a): l1 row selection
# ----------------------------------------------------------------------------

def num_selected(f: float, n: int) -> int:
    """k = ceil(f * n) rows, clamped to [1, n].

    Third-level paragraph of "Dion3: Full-Stack Orthogonal Updates": k = ceil(f n).
    """
    if not (0.0 < f <= 1.0):
        raise ValueError("fraction f must lie in (0, 1]")
    k = int(math.ceil(float(f) * float(n)))
    return max(1, min(n, k))


def accumulate(M: np.ndarray, G: np.ndarray) -> np.ndarray:
    """Error-feedback accumulation M <- M + G on every row, stored in fp32.

    The sum of two fp32 (or bf16-valued) numbers is formed exactly in double and
    rounded once to fp32, which is the fp32 round-to-nearest-even sum.
    """
    M64 = np.asarray(M, dtype=np.float32).astype(np.float64)
    G64 = np.asarray(G, dtype=np.float64)
    return (M64 + G64).astype(np.float32)


def row_l1(M: np.ndarray) -> np.ndarray:
    """l1 norm of each row, in double (third-level paragraph: rows picked by l1)."""
    return np.abs(np.asarray(M, dtype=np.float64)).sum(axis=1)


def row_sumsq(M: np.ndarray) -> np.ndarray:
    """Sum of squares of each row, in double."""
    M64 = np.asarray(M, dtype=np.float64)
    return (M64 * M64).sum(axis=1)


def select_rows(l1: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k rows with the largest l1 norm, ties to the lower index,
    returned in ascending order (int64)."""
    l1 = np.asarray(l1, dtype=np.float64)
    n = l1.shape[0]
    if not (1 <= k <= n):
        raise ValueError("k must lie in [1, n]")
    idx = np.arange(n)
    # Primary key: l1 descending; secondary: index ascending.
    order = np.lexsort((idx, -l1))
    return np.sort(order[:k])


# ----------------------------------------------------------------------------
# Step (b): orthogonalisation of the selected rows
# ----------------------------------------------------------------------------

def normalize(X: np.ndarray, eps: float) -> np.ndarray:
    """X / (||X||_F + eps) in double (reading: Frobenius normalisation)."""
    X64 = np.asarray(X, dtype=np.float64)
    return X64 / (math.sqrt(float((X64 * X64).sum())) + float(eps))


def newton_schulz(X: np.ndarray, coeffs=MUON_QUINTIC, steps: int = 5) -> np.ndarray:
    """Standard quintic Newton-Schulz applied directly to X (no Gram trick).

    Each iteration: A = X X^T, X <- a X + (b A + c A^2) X.  When X has more rows
    than columns the iteration runs on X^T and the result is transposed back.
    The first-level paragraph of "Dion3: Full-Stack Orthogonal Updates" states
    that Gram Newton-Schulz produces exactly this output.
    """
    a, b, c = (float(v) for v in coeffs)
    X = np.asarray(X, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    for _ in range(int(steps)):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


def gram_newton_schulz(X: np.ndarray, coeffs=MUON_QUINTIC, steps: int = 5,
                       restart_iter: int = 3, op_log: list | None = None) -> np.ndarray:
    """Gram Newton-Schulz in double, following the first-level paragraph of
    "Dion3: Full-Stack Orthogonal Updates": iterate on R = Y Y^T, accumulate the
    polynomial Q, restart once (recompute Y <- Q Y and R = Y Y^T) and multiply
    back O = Q Y at the end.

    Y is X, or X^T when X has more rows than columns (Gram matrix on the short
    side).  Iteration t (1-based):

      * if t == restart_iter (and t > 1): Y <- Q Y, R <- Y Y^T, Q <- I;
      * Z = a I + b R + c R^2;
      * Q <- Z if Q is the identity, else Q <- Z Q;
      * R <- Z R Z, unless t is the last iteration or the next one restarts.

    Used by the tests only, to pin the identity "Gram-NS equals standard NS" and
    the FLOP schedule; ``op_log`` (if given) receives one tuple per product:
    ("syrk", s, L), ("sym", s), ("rect", s, L).
    """
    a, b, c = (float(v) for v in coeffs)
    X = np.asarray(X, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    Y = X.T.copy() if tall else X.copy()
    s, L = Y.shape
    log = op_log if op_log is not None else []
    eye = np.eye(s)

    R = Y @ Y.T
    log.append(("syrk", s, L))
    Q = None  # None stands for the identity
    for t in range(1, int(steps) + 1):
        if t == restart_iter and t > 1:
            Y = Q @ Y
            log.append(("rect", s, L))
            R = Y @ Y.T
            log.append(("syrk", s, L))
            Q = None
        Z = a * eye + b * R + c * (R @ R)
        log.append(("sym", s))
        if Q is None:
            Q = Z
        else:
            Q = Z @ Q
            log.append(("sym", s))
        if t < steps and (t + 1) != restart_iter:
            R = Z @ (R @ Z)
            log.append(("sym", s))
            log.append(("sym", s))
    O = Q @ Y
    log.append(("rect", s, L))
    return O.T if tall else O


# ----------------------------------------------------------------------------
# Step (c): row-scatter update with error feedback
# ----------------------------------------------------------------------------

def round_to_fp32(x: np.ndarray) -> np.ndarray:
    """Round double values once to fp32 (RNE); returned as float64 values."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round double values once to bfloat16 (8 significant bits, RNE).

    Written from the format's definition (1 sign, 8 exponent, 7 fraction bits;
    subnormals below 2^-126 with spacing 2^-133); returned as float64 values.
    Rounding straight from double avoids the double rounding of going through
    fp32 first.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    finite = np.isfinite(x)
    xf = x[finite]
    mant, expo = np.frexp(xf)  # xf = mant * 2**expo, 0.5 <= |mant| < 1
    # Spacing of bf16 numbers around xf: 2**(expo - 8) for normals, fixed 2**-133
    # in the subnormal range (expo - 8 < -133).
    shift = np.maximum(expo - 8, -133).astype(np.float64)
    scaled = np.ldexp(xf, (-shift).astype(np.int64))
    r = np.ldexp(np.rint(scaled), shift.astype(np.int64))  # np.rint: half to even
    # Overflow: beyond the largest finite bf16 (rounded up) goes to infinity.
    big = np.abs(r) > 3.3895313892515355e38
    r[big] = np.sign(r[big]) * np.inf
    out[finite] = r
    out[~finite] = x[~finite]
    return out


def decay_rows(M: np.ndarray, S: np.ndarray, mu: float) -> np.ndarray:
    """Error feedback: M[S] <- fp32(mu * M[S]); other rows untouched.

    ``mu`` is used as its fp32 value (the kernel receives an fp32 mu)."""
    M = np.array(M, dtype=np.float32, copy=True)
    mu32 = float(np.float32(mu))
    M[S] = (mu32 * M[S].astype(np.float64)).astype(np.float32)
    return M


def update_rows(W: np.ndarray, S: np.ndarray, O: np.ndarray, lr_eff: float,
                param_dtype: str) -> np.ndarray:
    """W[S] <- round_p(W[S] - lr_eff * O), computed in double and rounded once to
    the parameter dtype ('f32' or 'bf16'); other rows untouched.  Values are
    returned as float64 arrays holding exactly representable numbers."""
    W = np.array(W, dtype=np.float64, copy=True)
    new = W[S] - float(lr_eff) * np.asarray(O, dtype=np.float64)
    if param_dtype == "bf16":
        W[S] = round_to_bf16(new)
    elif param_dtype == "f32":
        W[S] = round_to_fp32(new)
    else:
        raise ValueError("param_dtype must be 'f32' or 'bf16'")
    return W


def dion3_step(W: np.ndarray, M: np.ndarray, G: np.ndarray, *, f: float, mu: float,
               lr: float, eps: float = 1e-7, coeffs=MUON_QUINTIC, steps: int = 5,
               param_dtype: str = "bf16", lr_f32: bool = True,
               force_selection: np.ndarray | None = None):
    """One Dion3 step on one matrix (n x m), in the step order of the third-level
    paragraph of "Dion3: Full-Stack Orthogonal Updates":

      1. M <- M + G (all rows, fp32 storage);
      2. S = top-k rows of M by l1 norm, k = ceil(f n), ties to the lower index;
      3. X = M[S] / (||M[S]||_F + eps);
      4. O = standard quintic Newton-Schulz of X (equal to Gram-NS);
      5. W[S] <- round_p(W[S] - (lr / sqrt(f)) O);
      6. M[S] <- fp32(mu * M[S]).

    ``lr_f32`` rounds lr / sqrt(f) to fp32 (the value the kernel receives).
    ``force_selection`` replaces step 2's S (used by the parity harness only when
    the l1 gap at the k-th row lies within rounding of the GPU's fp32 sums).

    Returns (W_new as float64 values, M_new fp32, S int64, O float64).
    """
    n, _ = np.shape(M)
    M1 = accumulate(M, G)
    k = num_selected(f, n)
    if force_selection is None:
        S = select_rows(row_l1(M1), k)
    else:
        S = np.sort(np.asarray(force_selection, dtype=np.int64))
        assert S.shape == (k,)
    X = normalize(M1[S], eps)
    O = newton_schulz(X, coeffs, steps)
    lr_eff = float(lr) / math.sqrt(float(f))
    if lr_f32:
        lr_eff = float(np.float32(lr_eff))
    W1 = update_rows(W, S, O, lr_eff, param_dtype)
    M2 = decay_rows(M1, S, mu)
    return W1, M2, S, O


# ----------------------------------------------------------------------------
# NorMuon per-neuron normalisation (a reading; parity unpinned as to the pages)
# ----------------------------------------------------------------------------
# "Dion3 Cuts Muon Optimizer Time by Up to 6x ...", section "Dion3's fastest
# path is a combined systems stack": the per-neuron normalisation is inherited
# from NorMuon; "Dion3: Full-Stack Orthogonal Updates", limitations paragraph:
# it runs in float32.  Neither page defines it.  The reading, from the NorMuon
# method: a neuron is a row of W (an output unit); each row i keeps a running
# second moment v_i of the orthogonalised update's entries, the row is divided
# by sqrt(v_i) + eps, and the normalised update is rescaled to a fixed RMS.
# With row selection only the selected rows have an update, so only their v
# moves (as only their momentum decays), and the RMS is matched over the
# k x m block that is written.

def normuon_rows(O: np.ndarray, v_sel: np.ndarray, beta2: float, eps: float):
    """Per-row second moment and normalising factor of the orthogonalised rows.

    O: k x m (one row per selected parameter row), v_sel: the k selected rows'
    state.  v_i <- beta2 v_i + (1 - beta2) mean_j O_ij^2; d_i = 1 / (sqrt(v_i) +
    eps).  Returns (d, v_new) in float64 (the stored state is fp32(v_new))."""
    O = np.asarray(O, dtype=np.float64)
    ms = np.mean(O * O, axis=1)
    v_new = float(beta2) * np.asarray(v_sel, dtype=np.float64) + (1.0 - float(beta2)) * ms
    d = 1.0 / (np.sqrt(v_new) + float(eps))
    return d, v_new


def normuon_update(O: np.ndarray, d: np.ndarray, rms: float) -> np.ndarray:
    """The normalised update U = g * diag(d) O with g such that ||U||_F =
    rms * sqrt(k m) (U = 0 when diag(d) O = 0)."""
    On = np.asarray(O, dtype=np.float64) * np.asarray(d, dtype=np.float64)[:, None]
    F = float(np.sqrt(np.sum(On * On)))
    if F == 0.0:
        return np.zeros_like(On)
    return (float(rms) * math.sqrt(On.size) / F) * On


def dion3_step_normuon(W: np.ndarray, M: np.ndarray, G: np.ndarray, v: np.ndarray, *, f: float,
                       mu: float, lr: float, beta2: float = 0.95, nm_eps: float = 1e-8,
                       rms: float = 0.2, eps: float = 1e-7, coeffs=MUON_QUINTIC, steps: int = 5,
                       param_dtype: str = "bf16", lr_f32: bool = True,
                       force_selection: np.ndarray | None = None):
    """``dion3_step`` with the per-neuron normalisation between steps 4 and 5:
    v[S] <- fp32(beta2 v[S] + (1 - beta2) mean_j O^2), U = normuon_update(O,
    1 / (sqrt(v[S]) + nm_eps), rms), W[S] <- round_p(W[S] - (lr / sqrt(f)) U).
    v is the per-row fp32 state (length n); rows outside S keep theirs.

    Returns (W_new, M_new, S, O, v_new fp32)."""
    n, _ = np.shape(M)
    M1 = accumulate(M, G)
    k = num_selected(f, n)
    if force_selection is None:
        S = select_rows(row_l1(M1), k)
    else:
        S = np.sort(np.asarray(force_selection, dtype=np.int64))
        assert S.shape == (k,)
    X = normalize(M1[S], eps)
    O = newton_schulz(X, coeffs, steps)
    v_out = np.array(v, dtype=np.float32, copy=True)
    d, v_new = normuon_rows(O, v_out[S], beta2, nm_eps)
    v_out[S] = v_new.astype(np.float32)
    U = normuon_update(O, d, rms)
    lr_eff = float(lr) / math.sqrt(float(f))
    if lr_f32:
        lr_eff = float(np.float32(lr_eff))
    W1 = update_rows(W, S, U, lr_eff, param_dtype)
    M2 = decay_rows(M1, S, mu)
    return W1, M2, S, O, v_out
