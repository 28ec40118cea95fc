"""Float64 CPU oracle for the Dion / Orth-Dion optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` use it.  It shares no code with the CUDA path.

What it computes (junaidaliop.github.io "Orth-Dion", the update equations
and the symbol glossary under them):

    M_t     = G_t + R_t
    U_t     = orth(M_t V_{t-1})                    U in R^{m x r}
    W_t     = M_t^T U_t                            W in R^{n x r}
    Vbar_t  = orth(W_t)        (Orth-Dion)
            = colnorm(W_t)     (Dion: the same page notes that swapping
                                orth(W_t) for column normalisation gives
                                Dion; the Orth-Dion abstract on
                                thelatestinai.com 2605.16341 defines column
                                normalisation as scaling every column of the
                                right factor to length one)
    X_{t+1} = X_t - eta * s * U_t Vbar_t^T
    R_{t+1} = beta * (M_t - U_t (U_t^T M_t))
    V_t     = Vbar_t                               (warm start)

orth(.) is the orthonormal factor of a QR factorisation, i.e. an orthonormal
basis of the column space (same glossary).
Readings taken where the pages are silent:

* QR sign convention: thin QR whose triangular factor has a positive
  diagonal, which makes Q unique for a full-rank argument.
* Scale s: the pages print eta alone; the workloads add s, default
  sqrt(m / n).  s = 1 reproduces the printed equation exactly.
* U_t^T M_t equals W_t^T exactly, so the residual is written beta*(M - U W^T).
* Dion column with zero norm: stays zero (no epsilon anywhere).
* A rank-deficient argument of orth() (a QR diagonal entry below
  1e-12 * ||A||_F) is flagged, not repaired.

Every routine here is plain NumPy in float64, written to be checked by eye
against the equations above, with no blocking or reordering beyond them.
"""
from __future__ import annotations

import numpy as np

ORTH = "orth"   # Orth-Dion: Vbar = orth(W)
DION = "dion"   # Dion:      Vbar = colnorm(W)

RANK_TOL = 1e-12


def householder_qr_pos(A):
    """Thin QR of a tall matrix by Householder reflections, positive diagonal.

    Returns (Q, Rf): A = Q Rf with Q (m x k) having orthonormal columns and
    Rf (k x k) upper triangular with Rf[j, j] >= 0.

    This is orth(.) of the Orth-Dion glossary (the Q of a QR factorisation),
    in the textbook Householder form: reflector j maps the
    sub-column x = A[j:, j] to -sign(x_0) ||x|| e_1; Q is accumulated by
    applying the reflectors, in reverse order, to the first k columns of I;
    finally each column of Q (row of Rf) whose diagonal came out negative is
    negated.
    """
    A = np.array(A, dtype=np.float64, copy=True)
    m, k = A.shape
    if k > m:
        raise ValueError("thin QR needs rows >= columns")
    reflectors = []
    for j in range(k):
        x = A[j:, j]
        alpha = np.sqrt(np.dot(x, x))
        v = x.copy()
        v[0] += (1.0 if x[0] >= 0.0 else -1.0) * alpha
        vv = np.dot(v, v)
        if vv > 0.0:
            # A[j:, j:] <- (I - 2 v v^T / v^T v) A[j:, j:]
            A[j:, j:] -= np.outer(v, (2.0 / vv) * (v @ A[j:, j:]))
        reflectors.append((v, vv))
    Rf = np.triu(A[:k, :k])
    Q = np.eye(m, k)
    for j in reversed(range(k)):
        v, vv = reflectors[j]
        if vv > 0.0:
            Q[j:, :] -= np.outer(v, (2.0 / vv) * (v @ Q[j:, :]))
    d = np.where(np.diag(Rf) < 0.0, -1.0, 1.0)
    Q = Q * d[None, :]
    Rf = d[:, None] * Rf
    return Q, Rf


def lapack_qr_pos(A):
    """The same thin QR with a positive diagonal, with LAPACK's QR
    (numpy.linalg.qr, blocked Householder) as the factorisation step and the
    same sign fix: a library routine for the same definition, for arguments
    too large for the textbook loop above (an 8192 x 2048 argument takes
    minutes there).  Pinned against householder_qr_pos in the tests.
    """
    A = np.asarray(A, dtype=np.float64)
    if A.shape[1] > A.shape[0]:
        raise ValueError("thin QR needs rows >= columns")
    Q, Rf = np.linalg.qr(A, mode="reduced")
    d = np.where(np.diag(Rf) < 0.0, -1.0, 1.0)
    return Q * d[None, :], d[:, None] * Rf


def orth(A, qr=householder_qr_pos):
    """orth(A) with the positive-diagonal reading; returns (Q, deficient)."""
    A = np.asarray(A, dtype=np.float64)
    Q, Rf = qr(A)
    scale = np.linalg.norm(A)
    deficient = bool(np.any(np.abs(np.diag(Rf)) <= RANK_TOL * scale)) if scale > 0 else True
    return Q, deficient


def colnorm(W):
    """Dion's right factor: each column of W rescaled to unit Euclidean length.

    A column whose norm is exactly zero is left at zero.
    """
    W = np.asarray(W, dtype=np.float64)
    norms = np.sqrt(np.sum(W * W, axis=0))
    safe = np.where(norms > 0.0, norms, 1.0)
    return np.where(norms[None, :] > 0.0, W / safe[None, :], 0.0)


def default_scale(m, n):
    """s = sqrt(m / n), the reading used by every workload unless overridden."""
    return float(np.sqrt(m / n))


def oracle_step(X, G, R, V, eta, beta, variant=ORTH, scale=None, qr=householder_qr_pos):
    """One Dion / Orth-Dion step on one matrix, in float64.

    Inputs are widened exactly to float64 (fp32 and bf16 values are exactly
    representable).  Shapes: X, G, R are m x n; V (the warm start V_{t-1})
    is n x r.  ``scale=None`` means s = sqrt(m/n); ``qr`` is the thin-QR
    routine behind orth() (householder_qr_pos, or lapack_qr_pos for large
    arguments).  Returns a dict with the
    new state (X, R, V) and the intermediates M, P, U, W, Vbar plus a
    ``deficient`` flag (orth() met a rank-deficient argument).
    """
    X = np.asarray(X, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    m, n = X.shape
    r = V.shape[1]
    if G.shape != (m, n) or R.shape != (m, n) or V.shape != (n, r):
        raise ValueError("shape mismatch")
    if not (1 <= r <= min(m, n)):
        raise ValueError("need 1 <= r <= min(m, n)")
    s = default_scale(m, n) if scale is None else float(scale)

    M = G + R                                   # M_t = G_t + R_t
    P = M @ V                                   # M_t V_{t-1}
    U, def_u = orth(P, qr)                      # U_t = orth(M_t V_{t-1})
    W = M.T @ U                                 # W_t = M_t^T U_t
    if variant == ORTH:
        Vbar, def_w = orth(W, qr)               # Vbar_t = orth(W_t)
    elif variant == DION:
        Vbar, def_w = colnorm(W), False         # Vbar_t = colnorm(W_t)
    else:
        raise ValueError(f"unknown variant {variant!r}")
    X_new = X - eta * s * (U @ Vbar.T)          # X_{t+1} = X_t - eta s U_t Vbar_t^T
    R_new = beta * (M - U @ W.T)                # R_{t+1} = beta (M_t - U_t U_t^T M_t)
    return {
        "X": X_new, "R": R_new, "V": Vbar,      # V_t = Vbar_t
        "M": M, "P": P, "U": U, "W": W, "Vbar": Vbar,
        "deficient": def_u or def_w,
    }


def oracle_chain(X, R, V, grads, eta, beta, variant=ORTH, scale=None, qr=householder_qr_pos):
    """Run ``len(grads)`` chained steps in float64, each step's new X, R and V
    (V_t = Vbar_t) feeding the next; returns the list of step dicts."""
    out = []
    for G in grads:
        st = oracle_step(X, G, R, V, eta, beta, variant, scale, qr)
        X, R, V = st["X"], st["R"], st["V"]
        out.append(st)
    return out
