"""Float64 CPU oracle of the Dion3 row-selection step (test infrastructure only).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  The Dion3 abstract
(searcharxiv 2608.11612) changes Muon's update by orthogonalising only a
fraction of the momentum matrix's rows at each step; the selection rule is
not on the pages (parity unpinned beyond this reading):

    B <- mu B + G                                (Muon's momentum)
    S  = the k = ceil(rho m) rows of B with the largest Euclidean norm
         (ties: the lower row index), in increasing order
    Y  = ns_cubic(B[S], K)                       (muon_oracle: Y_0 = B[S] / ||B[S]||_F)
    X[S] <- X[S] - eta s Y;  the other rows of X are not changed
"""
from __future__ import annotations

import math

import numpy as np

from .muon_oracle import ns_cubic


def select_rows(B, k):
    """Indices of the k rows of B with the largest norm (ties: lower index), increasing."""
    norms = np.sum(np.asarray(B, dtype=np.float64) ** 2, axis=1)
    order = sorted(range(B.shape[0]), key=lambda i: (-norms[i], i))
    return np.array(sorted(order[:k]), dtype=np.int64)


def dion3_step(X, G, B, eta, mu, iters, row_fraction, scale=None, selected=None):
    """One step; ``selected`` overrides the selection (to follow another side's choice)."""
    X = np.array(X, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    m, n = X.shape
    s = math.sqrt(m / n) if scale is None else float(scale)
    B_new = mu * B + G
    k = min(m, max(1, math.ceil(row_fraction * m)))
    S = select_rows(B_new, k) if selected is None else np.asarray(selected, dtype=np.int64)
    Y = ns_cubic(B_new[S], iters)
    X[S] -= eta * s * Y
    return {"X": X, "B": B_new, "Y": Y, "selected": S}
