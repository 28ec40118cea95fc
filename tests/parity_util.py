"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the float64 oracle on exactly the stored values, compare."""
from __future__ import annotations

import numpy as np

from oracle import dion_oracle as O

# Tolerances (fixed by the specification of this path, not by the pages):
TOL_STEP = 1e-4      # relative Frobenius error of X and R after one step from identical state
TOL_CHAIN = 1e-3     # ... after 10 chained steps against the oracle's own float64 trajectory
TOL_ORTH = 1e-5      # max |U^T U - I|
TOL_DX = 1e-3        # relative Frobenius error of the update X_{t+1} - X_t (= -eta s U Vbar^T)


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def grad_to_device(g: np.ndarray, device):
    import torch
    if g.dtype == np.uint16:
        return torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(g, dtype=np.float32)).to(device)


def grad_f64(g) -> np.ndarray:
    return f64(g)


def orth_v0(V0_raw) -> np.ndarray:
    """V_0 = orth(N(0,1) draw), by the oracle's QR, rounded to fp32."""
    Q, _ = O.householder_qr_pos(np.asarray(V0_raw, dtype=np.float64))
    return Q.astype(np.float32)


def padded(t, ld):
    """A view of ``t`` (rows x cols) stored with a larger row pitch ``ld``."""
    import torch
    rows, cols = t.shape
    buf = torch.full((rows, ld), float("nan"), dtype=t.dtype, device=t.device)
    buf[:, :cols] = t
    return buf[:, :cols]


def state_snapshot(d):
    return {k: f64(d[k]) for k in ("X", "R", "V")}


def kappa(A) -> float:
    """2-norm condition number of a tall matrix (from the eigenvalues of A^T A)."""
    ev = np.linalg.eigvalsh(A.T @ A)
    return float(np.sqrt(ev[-1] / max(ev[0], 1e-300)))


def factor_tolerance(ref) -> float:
    """Relative error allowed on the right factor Vbar.

    A thin-QR factor moves by up to kappa times the relative perturbation of its
    argument, and the GPU's arguments carry fp32 rounding (2^-24): U = orth(P)
    by kappa(P), and Vbar = orth(W) (or W's unit columns) by kappa(W) on top of
    the error W inherits from U.  The bound is that sum, times 4, and never
    below the step tolerance."""
    return max(TOL_STEP, 4.0 * (kappa(ref["P"]) + kappa(ref["W"])) * 2.0 ** -24)


def check_step(before, G64, d_after, eta, beta, variant, scale=None, U_gpu=None, tol=TOL_STEP, qr=None):
    """Compare one GPU step (state ``before`` -> ``d_after``) with the oracle step
    from the same stored state: X and R (relative Frobenius error <= tol), the
    update X_{t+1} - X_t (<= TOL_DX), the new warm start V = Vbar (within
    factor_tolerance) and, when given, U^T U = I.  Returns the oracle's output
    and the errors."""
    kw = {} if qr is None else {"qr": qr}
    ref = O.oracle_step(before["X"], G64, before["R"], before["V"], eta, beta, variant, scale, **kw)
    after = state_snapshot(d_after)
    errs = {
        "X": rel(after["X"], ref["X"]),
        "R": rel(after["R"], ref["R"]),
        "dX": rel(after["X"] - before["X"], ref["X"] - before["X"]),
        "V": rel(after["V"], ref["V"]),
        "tol_V": factor_tolerance(ref),
    }
    if U_gpu is not None:
        U = f64(U_gpu)
        errs["UtU"] = float(np.abs(U.T @ U - np.eye(U.shape[1])).max())
    assert errs["X"] <= tol and errs["R"] <= tol, errs
    assert errs["dX"] <= TOL_DX, errs
    assert errs["V"] <= errs["tol_V"], errs
    if "UtU" in errs:
        assert errs["UtU"] <= TOL_ORTH, errs
    return ref, errs
