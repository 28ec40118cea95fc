"""Pins of the Muon comparator's float64 oracle (CPU only).

Each pin comes from mathematics the iteration must obey, computed
independently of the oracle: the singular-value map of the cubic iteration
against numpy's SVD, convergence to the polar factor, the closed form of the
momentum under a constant gradient, and planted slips that the pins catch.
"""
import numpy as np
import pytest

from oracle import muon_oracle as MU


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def spectral_pin(step, shape, iters, seed):
    """Y_K = U p^K(Sigma / ||B||_F) V^T for B = U Sigma V^T, p(s) = 1.5 s - 0.5 s^3."""
    g = rng(seed)
    m, n = shape
    X, G, B = g.standard_normal((m, n)), g.standard_normal((m, n)), g.standard_normal((m, n))
    out = step(X, G, B, 0.1, 0.9, iters, 1.3)
    Bn = 0.9 * B + G
    U, sv, Vt = np.linalg.svd(Bn, full_matrices=False)
    s = sv / np.sqrt(np.sum(sv ** 2))
    for _ in range(iters):
        s = 1.5 * s - 0.5 * s ** 3
    Y = (U * s[None, :]) @ Vt
    bad = []
    if np.abs(out["Y"] - Y).max() > 1e-12:
        bad.append("spectral map")
    if np.abs(out["X"] - (X - 0.1 * 1.3 * Y)).max() > 1e-12:
        bad.append("update")
    if np.abs(out["B"] - Bn).max() > 1e-13:
        bad.append("momentum")
    return bad


@pytest.mark.parametrize("shape", [(12, 7), (7, 12), (16, 16), (30, 5)])
@pytest.mark.parametrize("iters", [0, 1, 5])
def test_singular_value_map_matches_svd(shape, iters):
    assert spectral_pin(MU.muon_step, shape, iters, seed=shape[0] * 31 + iters) == []


def test_converges_to_polar_factor():
    """Singular values in [0.3, 1] of ||B||_F: many steps reach U V^T."""
    g = rng(3)
    m, n = 40, 25
    Ua, _ = np.linalg.qr(g.standard_normal((m, n)))
    Vb, _ = np.linalg.qr(g.standard_normal((n, n)))
    B = (Ua * np.linspace(1.0, 0.3, n)[None, :]) @ Vb.T
    Y = MU.ns_cubic(B, 40)
    assert np.abs(Y - Ua @ Vb.T).max() < 1e-12
    assert np.abs(Y.T @ Y - np.eye(n)).max() < 1e-12


def test_momentum_closed_form_under_constant_gradient():
    """B_0 = 0, G constant: B_t = G (1 - mu^t) / (1 - mu)."""
    g = rng(4)
    X, G = np.zeros((6, 4)), g.standard_normal((6, 4))
    B = np.zeros((6, 4))
    for t in range(1, 6):
        B = MU.muon_step(X, G, B, 0.0, 0.8, 1)["B"]
        assert np.abs(B - G * (1 - 0.8 ** t) / (1 - 0.8)).max() < 1e-13


def _mutant(kind):
    def step(X, G, B, eta, mu, iters, scale=None):
        X, G, B = (np.asarray(a, dtype=np.float64) for a in (X, G, B))
        m, n = X.shape
        s = np.sqrt(m / n) if scale is None else scale
        Bn = (B + mu * G) if kind == "momentum_swapped" else mu * B + G
        nrm = np.linalg.norm(Bn, 2) if kind == "spectral_norm" else np.linalg.norm(Bn)
        Y = Bn if kind == "no_normalisation" else Bn / nrm
        for _ in range(iters + (1 if kind == "extra_iteration" else 0)):
            if kind == "coefficient_sign":
                Y = 1.5 * Y + 0.5 * ((Y @ Y.T) @ Y)
            elif kind == "coefficients_swapped":
                Y = 0.5 * Y - 1.5 * ((Y @ Y.T) @ Y)
            else:
                Y = 1.5 * Y - 0.5 * ((Y @ Y.T) @ Y)
        Xn = X + eta * s * Y if kind == "update_sign" else X - eta * s * Y
        return {"X": Xn, "B": Bn, "Y": Y}
    return step


MUTANTS = ["momentum_swapped", "spectral_norm", "no_normalisation", "extra_iteration",
           "coefficient_sign", "coefficients_swapped", "update_sign"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistakes_are_caught(kind):
    assert spectral_pin(_mutant(kind), (12, 7), 3, seed=9), kind
    assert spectral_pin(_mutant("none"), (12, 7), 3, seed=9) == []
