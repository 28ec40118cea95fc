"""Float64 CPU oracle of the low-rank Muon variant (test infrastructure only).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  The low-rank
orthogonalisation abstract quoted on thelatestinai.com (the listing of
2605.16341) says only that low-rank Muon orthogonalises by exploiting the low
rank of gradients; the pages give no algorithm (parity unpinned beyond the
reading below).  The reading of this library, built from the pages' own
pieces: Muon's momentum (Dion3 abstract: Muon orthogonalises the momentum),
a fresh Gaussian sketch in place of Dion's warm start, and the Orth-Dion
right factor (junaidaliop.github.io "Orth-Dion": orth() = QR of the column
space, positive diagonal):

    M = G + mu B                 (momentum, B its previous value)
    U = orth(M Omega)            (Omega: n x r Gaussian, drawn fresh by the caller)
    W = M^T U,  Vbar = orth(W)
    X <- X - eta s U Vbar^T,  B <- M
"""
from __future__ import annotations

import numpy as np

from .dion_oracle import default_scale, householder_qr_pos, orth


def lowrank_muon_step(X, G, B, Omega, eta, mu, scale=None, qr=householder_qr_pos):
    X, G, B, Omega = (np.asarray(a, dtype=np.float64) for a in (X, G, B, Omega))
    m, n = X.shape
    s = default_scale(m, n) if scale is None else float(scale)
    M = G + mu * B
    U = orth(M @ Omega, qr)[0]
    W = M.T @ U
    Vbar = orth(W, qr)[0]
    return {"X": X - eta * s * (U @ Vbar.T), "B": M, "U": U, "W": W, "Vbar": Vbar, "V": Vbar}
