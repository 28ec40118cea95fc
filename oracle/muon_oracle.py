"""Float64 CPU oracle for the Muon comparator step (Newton-Schulz orthogonalisation).

TEST INFRASTRUCTURE ONLY: like dion_oracle, only ``tests/``, the smoke check
and the bench's CPU legs may import it; it shares no code with the CUDA path.

The pages describe Muon only in words: it orthogonalises the momentum of each
weight matrix with a Newton-Schulz iteration whose cost is cubic in the
matrix size (searcharxiv 2608.11612 "Dion3" abstract; the artiverse.ca post
"What Made Muon Stand Out"; the Dion abstract on searcharxiv 2504.05295).  They
print neither the momentum rule, the iteration's coefficients nor its length.
Readings taken here (the plainest ones the pages support):

* momentum:      B_t = mu B_{t-1} + G_t
* normalisation: Y_0 = B_t / ||B_t||_F        (every singular value in (0, 1])
* iteration:     Y_{k+1} = 1.5 Y_k - 0.5 Y_k Y_k^T Y_k,  k = 0 .. K-1
                 (the textbook cubic Newton-Schulz iteration for the polar
                 factor; it maps every singular value s to 1.5 s - 0.5 s^3 and
                 keeps the singular vectors)
* update:        X_{t+1} = X_t - eta s Y_K     (s = sqrt(m / n), as for Dion)

Plain NumPy, in the order above; Y Y^T Y is formed as (Y Y^T) Y, one of the two
equal groupings.
"""
from __future__ import annotations

import numpy as np


def ns_cubic(B, iters):
    """K steps of the cubic Newton-Schulz iteration from Y_0 = B / ||B||_F."""
    B = np.asarray(B, dtype=np.float64)
    nrm = np.linalg.norm(B)
    Y = B / nrm if nrm > 0 else np.zeros_like(B)
    for _ in range(iters):
        Y = 1.5 * Y - 0.5 * ((Y @ Y.T) @ Y)
    return Y


def muon_step(X, G, B, eta, mu, iters, scale=None):
    """One Muon step on one matrix; returns dict(X, B, Y)."""
    X = np.asarray(X, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    m, n = X.shape
    s = float(np.sqrt(m / n)) if scale is None else float(scale)
    B_new = mu * B + G                          # momentum
    Y = ns_cubic(B_new, iters)                  # orthogonalised momentum
    return {"X": X - eta * s * Y, "B": B_new, "Y": Y}
