"""Float64 backend of the row-sharded Dion / Orth-Dion step (test infrastructure).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  One rank's share of
the step of the Orth-Dion update equations (junaidaliop.github.io
"Orth-Dion") when the rows of X, G and R are split over ranks and V is
replicated, cut at the same exchange points as the library's staged step:

  stage 0  M_p = G_p + R_p, P_p = M_p V, exchange S = P_p^T P_p
  stage 1  S (summed over ranks) = Rc^T Rc (Cholesky, positive diagonal),
           Q_p = P_p Rc^-1, exchange S = Q_p^T Q_p
  stage 2  S = Rc2^T Rc2, U_p = Q_p Rc2^-1, exchange S = 0 (no third pass in float64)
  stage 3  exchange W = M_p^T U_p
  stage 4  Vbar = orth(W) or colnorm(W) (replicated), X_p -= eta s U_p Vbar^T,
           R_p = beta (M_p - U_p W^T), V = Vbar

Two CholeskyQR passes on the summed Gram give the thin-QR factor of the
stacked P with a positive diagonal (to float64 rounding for the condition
numbers used here), i.e. the same U as dion_oracle's Householder orth() of
the whole P; the tests check that.  The exchange buffers are float64 torch
tensors so that a torch.distributed process group can sum them.
"""
from __future__ import annotations

import numpy as np

from .dion_oracle import ORTH, colnorm, orth


class ShardBackend:
    def __init__(self, X, G, R, V, eta, beta, variant=ORTH, scale=1.0):
        self.X = np.array(X, dtype=np.float64)
        self.G = np.asarray(G, dtype=np.float64)
        self.R = np.array(R, dtype=np.float64)
        self.V = np.array(V, dtype=np.float64)
        self.eta, self.beta, self.variant, self.scale = eta, beta, variant, scale
        import torch
        r = self.V.shape[1]
        self._gram = torch.zeros((r, r), dtype=torch.float64)
        self._w = torch.zeros(self.V.shape, dtype=torch.float64)

    def exchange(self, name):
        return self._gram if name == "gram" else self._w

    def _chol_inv(self):
        S = self._gram.numpy()
        L = np.linalg.cholesky(S)          # S = L L^T, positive diagonal; Rc = L^T
        return np.linalg.inv(L.T)

    def stage(self, k):
        import torch
        if k == 0:
            self.M = self.G + self.R
            self.P = self.M @ self.V
            self._gram.copy_(torch.from_numpy(self.P.T @ self.P))
        elif k == 1:
            self.Q = self.P @ self._chol_inv()
            self._gram.copy_(torch.from_numpy(self.Q.T @ self.Q))
        elif k == 2:
            self.U = self.Q @ self._chol_inv()
            self._gram.zero_()
        elif k == 3:
            self._w.copy_(torch.from_numpy(self.M.T @ self.U))
        elif k == 4:
            W = self._w.numpy()
            Vbar = orth(W)[0] if self.variant == ORTH else colnorm(W)
            self.X = self.X - self.eta * self.scale * (self.U @ Vbar.T)
            self.R = self.beta * (self.M - self.U @ W.T)
            self.V = Vbar
            self.W = W
