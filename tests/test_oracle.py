"""Pins for the float64 oracle, checked against things other than itself.

The pages print no worked example, so the oracle is pinned by:
  * an independent QR algorithm (modified Gram-Schmidt with
    re-orthogonalisation) and exact rational/surd Gram-Schmidt (sympy),
  * library special cases (numpy SVD projectors, polar factors, singular
    subspaces),
  * closed forms and invariants that follow from the update equations on
    junaidaliop.github.io "Orth-Dion" (update equations and glossary) and the
    Dion column-normalisation rule of the Orth-Dion abstract
    (thelatestinai.com 2605.16341).
A final test plants mistakes in copies of the oracle and checks that these
pins catch every one of them.
"""
import math

import numpy as np
import pytest

from oracle import dion_oracle as O
from rank_orthonormalized_optimizer_03_b300 import synth, workloads


def rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


# ------------------------------------------------------------- QR ----------
def mgs_reorth(A):
    """Independent thin QR: modified Gram-Schmidt, two passes per column."""
    A = np.array(A, dtype=np.float64)
    m, k = A.shape
    Q = np.zeros((m, k))
    for j in range(k):
        v = A[:, j].copy()
        for _ in range(2):
            for i in range(j):
                v -= (Q[:, i] @ v) * Q[:, i]
        Q[:, j] = v / np.linalg.norm(v)
    return Q


@pytest.mark.parametrize("shape", [(7, 3), (50, 7), (200, 30), (16, 16), (64, 1)])
def test_householder_orthonormal_reconstructs_positive(shape):
    A = rng(1).standard_normal(shape)
    Q, Rf = O.householder_qr_pos(A)
    k = shape[1]
    assert Q.shape == shape and Rf.shape == (k, k)
    assert np.abs(Q.T @ Q - np.eye(k)).max() < 1e-13
    assert np.abs(Q @ Rf - A).max() < 1e-13 * max(1.0, np.abs(A).max()) * k
    assert np.all(np.diag(Rf) > 0)
    assert np.abs(np.tril(Rf, -1)).max() == 0.0


@pytest.mark.parametrize("shape", [(9, 4), (40, 12), (120, 33)])
def test_householder_equals_mgs_reorth(shape):
    A = rng(2).standard_normal(shape)
    Q, _ = O.householder_qr_pos(A)
    assert np.abs(Q - mgs_reorth(A)).max() < 1e-12


def test_householder_exact_gram_schmidt_sympy():
    sympy = pytest.importorskip("sympy")
    A = sympy.Matrix([[2, -1, 0], [1, 3, -2], [0, 1, 4], [-2, 0, 1], [1, 1, 1]])
    cols = []
    for j in range(A.shape[1]):
        v = A[:, j]
        for q in cols:
            v = v - (q.dot(A[:, j])) * q
        cols.append(sympy.simplify(v / sympy.sqrt(v.dot(v))))
    Qx = np.array([[float(c[i]) for c in cols] for i in range(A.shape[0])])
    Q, Rf = O.householder_qr_pos(np.array(A.tolist(), dtype=np.float64))
    assert np.abs(Q - Qx).max() < 1e-14
    # R = Q^T A exactly: first diagonal entry is ||a_1|| = sqrt(10)
    assert abs(Rf[0, 0] - math.sqrt(10.0)) < 1e-14


def test_householder_projector_matches_svd():
    A = rng(3).standard_normal((60, 9))
    Q, _ = O.householder_qr_pos(A)
    Us, _, _ = np.linalg.svd(A, full_matrices=False)
    assert np.abs(Q @ Q.T - Us @ Us.T).max() < 1e-13


def test_householder_sign_special_cases():
    # negated identity block: Q = -I, R = I under the positive-diagonal reading
    A = np.vstack([-np.eye(3), np.zeros((2, 3))])
    Q, Rf = O.householder_qr_pos(A)
    assert np.abs(Q - A).max() < 1e-15 and np.abs(Rf - np.eye(3)).max() < 1e-15
    # already-orthogonal columns with mixed signs: Q = A D, R = diag(|.|)
    B = np.array([[0.0, 3.0], [-2.0, 0.0], [0.0, 0.0]])
    Q, Rf = O.householder_qr_pos(B)
    assert np.abs(Q - np.array([[0, 1.0], [-1.0, 0], [0, 0]])).max() < 1e-15
    assert np.abs(Rf - np.diag([2.0, 3.0])).max() < 1e-15


def test_orth_flags_rank_deficiency():
    A = rng(4).standard_normal((30, 3))
    A = np.hstack([A, A[:, :1] * 2.0])
    _, deficient = O.orth(A)
    assert deficient
    _, ok = O.orth(rng(4).standard_normal((30, 4)))
    assert not ok


def test_colnorm_unit_columns_and_zero_column():
    W = rng(5).standard_normal((20, 5))
    W[:, 2] = 0.0
    C = O.colnorm(W)
    nrm = np.linalg.norm(C, axis=0)
    assert np.allclose(nrm[[0, 1, 3, 4]], 1.0, atol=1e-15) and nrm[2] == 0.0
    # direction is preserved
    assert np.abs(C[:, 0] * np.linalg.norm(W[:, 0]) - W[:, 0]).max() < 1e-15


# ------------------------------------------------------------- step invariants
def random_state(m, n, r, seed, r_nonzero=True):
    g = rng(seed)
    X = g.normal(0, 0.02, (m, n))
    G = g.standard_normal((m, 3)) @ g.standard_normal((3, n)) + 0.1 * g.standard_normal((m, n))
    R = 0.05 * g.standard_normal((m, n)) if r_nonzero else np.zeros((m, n))
    V = g.standard_normal((n, r))
    return X, G, R, V


def step_violations(step, X, G, R, V, eta, beta, variant, scale=None):
    """All invariant checks of one step; returns the names of the failing ones."""
    m, n = X.shape
    r = V.shape[1]
    s = math.sqrt(m / n) if scale is None else scale
    out = step(X, G, R, V, eta, beta, variant, scale)
    M = G + R
    U, Vb, W = out["U"], out["Vbar"], out["W"]
    dX = out["X"] - X
    bad = []

    def chk(name, ok):
        if not ok:
            bad.append(name)

    chk("U_orthonormal", np.abs(U.T @ U - np.eye(r)).max() < 1e-12)
    # U spans col(M V) and U^T (M V) is upper triangular with positive diagonal
    T = U.T @ (M @ V)
    chk("U_spans_MV", np.abs(M @ V - U @ T).max() < 1e-10 * max(1, np.abs(M @ V).max()))
    chk("U_posdiag_triangular", np.all(np.diag(T) > 0) and np.abs(np.tril(T, -1)).max() < 1e-10)
    # residual: R' = beta (I - U U^T) M  <=>  U^T R' = 0 and R' + beta U U^T M = beta M
    Rn = out["R"]
    chk("residual_orth_U", np.abs(U.T @ Rn).max() < 1e-10 * max(1, np.abs(M).max()) * max(m, n))
    chk("energy_identity", abs(np.sum(Rn ** 2) - beta ** 2 * (np.sum(M ** 2) - np.sum(W ** 2)))
        < 1e-10 * max(1.0, np.sum(M ** 2)))
    chk("residual_plus_projection", np.abs(Rn + beta * U @ (U.T @ M) - beta * M).max()
        < 1e-10 * max(1, np.abs(M).max()))
    # X update: -dX/(eta s) = U Vbar^T with ||.||_F^2 = r (D2); descent direction
    chk("dX_norm", abs(np.linalg.norm(dX) - eta * s * math.sqrt(r)) < 1e-10 * max(1, eta * s * math.sqrt(r)))
    Vrec = -(dX.T @ U) / (eta * s)
    chk("dX_rank_r_in_U", np.abs(dX - U @ (U.T @ dX)).max() < 1e-12)
    chk("dX_descent", np.sum(dX * M) < 0)
    if variant == O.ORTH:
        chk("Vbar_orthonormal", np.abs(Vrec.T @ Vrec - np.eye(r)).max() < 1e-10)
        TW = Vrec.T @ W
        chk("Vbar_posdiag_triangular", np.all(np.diag(TW) > 0) and np.abs(np.tril(TW, -1)).max() < 1e-9)
        chk("Vbar_spans_W", np.abs(W - Vrec @ TW).max() < 1e-9 * max(1, np.abs(W).max()))
        chk("spectral_norm_one", abs(np.linalg.norm(Vrec, 2) - 1.0) < 1e-10)
    else:
        nrm = np.linalg.norm(Vrec, axis=0)
        chk("Vbar_unit_columns", np.abs(nrm - 1.0).max() < 1e-10)
        chk("Vbar_parallel_W", np.abs(Vrec * np.linalg.norm(W, axis=0) - W).max()
            < 1e-9 * max(1, np.abs(W).max()))
        sn = np.linalg.norm(Vrec, 2)
        chk("spectral_norm_range", 1 - 1e-10 <= sn <= math.sqrt(r) + 1e-10)
    chk("warm_start_is_Vbar", np.abs(out["V"] - Vrec).max() < 1e-10)
    return bad


CASES = [(40, 24, 5), (24, 40, 5), (64, 64, 1), (33, 17, 17), (17, 33, 17), (128, 96, 12)]


@pytest.mark.parametrize("variant", [O.ORTH, O.DION])
@pytest.mark.parametrize("m,n,r", CASES)
def test_step_invariants(m, n, r, variant):
    X, G, R, V = random_state(m, n, r, seed=m * 7 + n + r)
    assert step_violations(O.oracle_step, X, G, R, V, 0.01, 0.95, variant) == []
    # explicit scale, beta = 0 and beta = 1 corners
    assert step_violations(O.oracle_step, X, G, R, V, 0.3, 0.0, variant, scale=1.0) == []
    assert step_violations(O.oracle_step, X, G, R, V, 0.3, 1.0, variant, scale=2.5) == []


def test_rank_one_closed_form():
    """r = 1 (D4): u = Mv/||Mv||, w = M^T u, vbar = w/||w||; both variants agree."""
    X, G, R, V = random_state(30, 20, 1, seed=11)
    M = G + R
    u = M @ V[:, 0]
    u = u / np.linalg.norm(u)
    w = M.T @ u
    vb = w / np.linalg.norm(w)
    for variant in (O.ORTH, O.DION):
        out = O.oracle_step(X, G, R, V, 0.1, 0.9, variant, scale=1.0)
        assert np.abs(out["U"][:, 0] - u).max() < 1e-13
        assert np.abs(out["Vbar"][:, 0] - vb).max() < 1e-13
        assert np.abs(out["X"] - (X - 0.1 * np.outer(u, vb))).max() < 1e-14
        assert np.abs(out["R"] - 0.9 * (M - np.outer(u, w))).max() < 1e-13


def test_exact_rank_aligned_gives_polar_factor():
    """rank(M) <= r and V_prev = B (signed permutation): U Vbar^T = polar(M) (D5)."""
    g = rng(12)
    m, n, r = 12, 9, 4
    A, _ = np.linalg.qr(g.standard_normal((m, r)))
    B, _ = np.linalg.qr(g.standard_normal((n, r)))
    M = A @ np.diag([5.0, 3.0, 2.0, 0.5]) @ B.T
    Vp = B[:, [2, 0, 3, 1]] * np.array([1, -1, -1, 1])
    out = O.oracle_step(np.zeros((m, n)), M, np.zeros((m, n)), Vp, 1.0, 1.0, O.ORTH, scale=1.0)
    Us, ss, Vst = np.linalg.svd(M)
    polar = Us[:, :r] @ Vst[:r]
    assert np.abs(out["U"] @ out["Vbar"].T - polar).max() < 1e-12
    assert np.abs(out["R"]).max() < 1e-12


def test_exact_rank_spanning_partial_isometry():
    """V_prev only spanning row(M): residual 0, U Vbar^T a partial isometry (D5)."""
    g = rng(13)
    m, n, r = 11, 8, 3
    A, _ = np.linalg.qr(g.standard_normal((m, r)))
    B, _ = np.linalg.qr(g.standard_normal((n, r)))
    M = A @ np.diag([4.0, 2.0, 1.0]) @ B.T
    Vp = B @ g.standard_normal((r, r))
    out = O.oracle_step(np.zeros((m, n)), M, np.zeros((m, n)), Vp, 1.0, 1.0, O.ORTH, scale=1.0)
    Pm = out["U"] @ out["Vbar"].T
    sv = np.linalg.svd(Pm, compute_uv=False)
    assert np.abs(out["R"]).max() < 1e-12
    assert np.abs(sv[:r] - 1.0).max() < 1e-12 and np.abs(sv[r:]).max() < 1e-12
    assert np.abs(A @ A.T @ out["U"] - out["U"]).max() < 1e-12          # col space
    assert np.abs(out["Vbar"] - B @ (B.T @ out["Vbar"])).max() < 1e-12  # row space
    nuc = np.linalg.svd(M, compute_uv=False).sum()
    assert np.trace(M.T @ Pm) <= nuc + 1e-12


def fixed_gradient_pin(chain):
    """G fixed, beta = 0, through a chain function: V_t follows subspace
    iteration on G^T G (D6), converging to the top-r right singular subspace
    at (sigma_{r+1}/sigma_r)^2 per step.  Returns the list of failures."""
    g = rng(14)
    m, n, r = 50, 30, 4
    Ua, _ = np.linalg.qr(g.standard_normal((m, n)))
    Vb, _ = np.linalg.qr(g.standard_normal((n, n)))
    svals = np.concatenate([[10.0, 9.0, 8.0, 7.0], np.linspace(3.5, 0.5, n - 4)])
    G = Ua @ np.diag(svals) @ Vb.T
    V = g.standard_normal((n, r))
    X, R = np.zeros((m, n)), np.zeros((m, n))
    top = Vb[:, :r]
    rate = (svals[r] / svals[r - 1]) ** 2
    steps = chain(X, R, V, [G] * 12, 0.0, 0.0, O.ORTH, 1.0)
    errs = [np.linalg.norm(top @ top.T - st["V"] @ st["V"].T, 2) for st in steps]
    bad = []
    if not errs[-1] < 1e-4:
        bad.append(f"no convergence: {errs[-1]:.3g}")
    # geometric decay at (sigma_{r+1}/sigma_r)^2 per step, up to a constant
    for a, b in zip(errs[3:-1], errs[4:]):
        if not b <= a * rate * 1.05:
            bad.append(f"decay {b / a:.3g} > {rate:.3g}")
            break
    return bad


def deflation_pin(chain):
    """G = 0, beta = 1, through a chain function: successive U_t are mutually
    orthogonal, the residual energy falls by ||W_t||^2 per step (D6, D3) and
    X collects every step's -eta s U_t Vbar_t^T, which holds only if every step
    reads the previous step's X, R and V."""
    g = rng(15)
    m, n, r = 40, 30, 3
    R0 = g.standard_normal((m, n))
    V = g.standard_normal((n, r))
    X = np.zeros((m, n))
    steps = chain(X, R0, V, [np.zeros((m, n))] * 4, 0.1, 1.0, O.ORTH, 1.0)
    bad = []
    # X carried: X_T = X_0 - eta s sum_t U_t Vbar_t^T
    X_sum = X - 0.1 * sum(st["U"] @ st["Vbar"].T for st in steps)
    if np.abs(steps[-1]["X"] - X_sum).max() >= 1e-12:
        bad.append("X not accumulated across steps")
    e_prev = np.sum(R0 ** 2)
    for t, st in enumerate(steps):
        e = np.sum(st["R"] ** 2)
        if abs(e - (e_prev - np.sum(st["W"] ** 2))) >= 1e-10 * e_prev:
            bad.append(f"energy identity fails at step {t}")
        e_prev = e
        for j in range(t):
            if np.abs(st["U"].T @ steps[j]["U"]).max() >= 1e-12:
                bad.append(f"U_{t} not orthogonal to U_{j}")
    return bad


def test_fixed_gradient_converges_to_top_subspace():
    assert fixed_gradient_pin(O.oracle_chain) == []


def test_zero_gradient_deflates():
    assert deflation_pin(O.oracle_chain) == []


def _chain_mutant(kind):
    """oracle_chain with one plausible slip in how the state is carried."""
    def chain(X, R, V, grads, eta, beta, variant=O.ORTH, scale=None):
        out = []
        R0, V0 = R, V
        for G in grads:
            st = O.oracle_step(X, G, R, V, eta, beta, variant, scale)
            X = X if kind == "X_not_carried" else st["X"]
            R = R0 if kind == "R_not_carried" else st["R"]
            V = {"V_not_carried": V0, "V_from_P": st["P"][: V0.shape[0]]}.get(kind, st["V"])
            out.append(st)
        return out
    return chain


# (Carrying W instead of Vbar = orth(W) is not among them: orth(M W) = orth(M orth(W))
# because W's triangular factor has a positive diagonal, so that chain is the same
# computation for Orth-Dion, not a slip.)
CHAIN_MUTANTS = ["X_not_carried", "R_not_carried", "V_not_carried", "V_from_P"]


@pytest.mark.parametrize("kind", CHAIN_MUTANTS)
def test_planted_chain_mistakes_are_caught(kind):
    """A chain that drops or mis-carries R or V fails one of the chain pins."""
    mutant = _chain_mutant(kind)
    assert fixed_gradient_pin(mutant) or deflation_pin(mutant), kind


def test_lapack_qr_equals_householder():
    """The library-routine QR (used for the largest parity cases) and the
    textbook Householder QR compute the same positive-diagonal factors."""
    g = rng(23)
    for shape in [(300, 40), (97, 97), (512, 3)]:
        A = g.standard_normal(shape)
        Qh, Rh = O.householder_qr_pos(A)
        Ql, Rl = O.lapack_qr_pos(A)
        assert np.abs(Qh - Ql).max() < 1e-11 and np.abs(Rh - Rl).max() < 1e-10
    X, G, R, V = random_state(60, 40, 6, seed=24)
    a = O.oracle_step(X, G, R, V, 0.01, 0.9, O.ORTH)
    b = O.oracle_step(X, G, R, V, 0.01, 0.9, O.ORTH, qr=O.lapack_qr_pos)
    for k in ("X", "R", "V", "U", "W"):
        assert np.abs(a[k] - b[k]).max() < 1e-11, k


def test_variants_share_U_R_W_trajectory():
    """Dion and Orth-Dion differ only in X (D1)."""
    m, n, r = 40, 24, 5
    X, _, _, V = random_state(m, n, r, seed=16)
    grads = [random_state(m, n, r, seed=100 + t)[1] for t in range(8)]
    a = O.oracle_chain(X, np.zeros((m, n)), V, grads, 0.01, 0.95, O.ORTH)
    b = O.oracle_chain(X, np.zeros((m, n)), V, grads, 0.01, 0.95, O.DION)
    for sa, sb in zip(a, b):
        assert np.abs(sa["U"] - sb["U"]).max() < 1e-10
        assert np.abs(sa["R"] - sb["R"]).max() < 1e-10
        assert np.abs(sa["W"] - sb["W"]).max() < 1e-10
    assert np.abs(a[-1]["X"] - b[-1]["X"]).max() > 1e-6


def test_default_scale_and_rank_deficient_flag():
    X, G, R, V = random_state(32, 8, 3, seed=17)
    a = O.oracle_step(X, G, R, V, 0.01, 0.9, O.ORTH)
    b = O.oracle_step(X, G, R, V, 0.01, 0.9, O.ORTH, scale=2.0)
    assert np.abs(a["X"] - b["X"]).max() == 0.0           # sqrt(32/8) = 2
    z = np.zeros((32, 8))
    assert O.oracle_step(X, z, z, V, 0.01, 0.9, O.ORTH)["deficient"]
    assert not a["deficient"]


def test_bad_arguments_raise():
    X, G, R, V = random_state(10, 6, 2, seed=18)
    with pytest.raises(ValueError):
        O.oracle_step(X, G[:, :5], R, V, 0.1, 0.9)
    with pytest.raises(ValueError):
        O.oracle_step(X, G, R, np.zeros((6, 7)), 0.1, 0.9)
    with pytest.raises(ValueError):
        O.oracle_step(X, G, R, V, 0.1, 0.9, variant="muon")


# ------------------------------------------------------------- generators
def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(bits)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 tie -> 1+2^-6 (even); 1+2^-9 rounds down
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]


def test_host_inputs_deterministic_and_shaped():
    wl = workloads.single_256x128()
    a = synth.host_inputs(wl, seed=0)
    b = synth.host_inputs(wl, seed=0)
    assert a.X0.dtype == np.float32 and a.X0.shape == (256, 128)
    assert len(a.grads) == 10 and a.grads[0].dtype == np.float32
    assert np.array_equal(a.grads[3], b.grads[3]) and np.array_equal(a.V0_raw, b.V0_raw)
    wl2 = workloads.square_1024()
    c = synth.host_inputs(wl2, seed=0, steps=1)
    assert c.grads[0].dtype == np.uint16
    gs = c.grad_f64(0)
    # A B^T with A, B ~ N(0,1)/sqrt(32): entry variance 32 * (1/32)^2 = 1/32; plus 0.05^2 noise
    assert abs(gs.std() - math.sqrt(1 / 32 + 0.05 ** 2)) < 0.01


# ------------------------------------------------------------- planted mistakes
def _mutant(kind):
    def step(X, G, R, V, eta, beta, variant=O.ORTH, scale=None):
        Xf, Gf, Rf, Vf = (np.asarray(a, dtype=np.float64) for a in (X, G, R, V))
        m, n = Xf.shape
        s = O.default_scale(m, n) if scale is None else scale
        M = Gf - Rf if kind == "M_sign" else (Gf if kind == "M_drop_R" else Gf + Rf)
        P = M @ Vf
        if kind == "U_no_signfix":
            U, _ = np.linalg.qr(P)
            U = -U
        else:
            U, _ = O.orth(P)
        W = (M @ U[: n] if kind == "W_no_transpose" and m == n else M.T @ U)
        if kind == "W_wrong_factor":
            W = M.T @ (M @ Vf)
        if variant == O.ORTH:
            Vb = O.orth(W)[0] if kind != "Vbar_colnorm" else O.colnorm(W)
        else:
            Vb = O.colnorm(W) if kind != "Vbar_colnorm" else O.orth(W)[0]
        if kind == "Vbar_unnormalised":
            Vb = W
        step_ = -1.0 if kind == "X_sign" else 1.0
        sc = 1.0 if kind == "X_drop_scale" else s
        Xn = Xf - step_ * eta * sc * (U @ Vb.T)
        if kind == "X_transposed_factor" and m == n:
            Xn = Xf - eta * sc * (Vb @ U.T)
        b = 1.0 if kind == "R_drop_beta" else beta
        Rn = b * (M - U @ W.T) if kind != "R_sign" else b * (M + U @ W.T)
        if kind == "R_no_projection":
            Rn = b * M
        Vn = Vf if kind == "V_not_updated" else Vb
        return {"X": Xn, "R": Rn, "V": Vn, "M": M, "P": P, "U": U, "W": W, "Vbar": Vb,
                "deficient": False}
    return step


MUTANTS = ["M_sign", "M_drop_R", "U_no_signfix", "W_no_transpose", "W_wrong_factor",
           "Vbar_colnorm", "Vbar_unnormalised", "X_sign", "X_drop_scale",
           "X_transposed_factor", "R_drop_beta", "R_sign", "R_no_projection", "V_not_updated"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistakes_are_caught(kind):
    """Every plausible slip in the step fails at least one pin above."""
    caught = False
    for (m, n, r) in [(24, 24, 4), (40, 24, 5)]:
        X, G, R, V = random_state(m, n, r, seed=19)
        for variant in (O.ORTH, O.DION):
            if step_violations(_mutant(kind), X, G, R, V, 0.01, 0.95, variant):
                caught = True
    assert caught, kind
    # and the unmutated copy passes (so the harness itself is sound)
    X, G, R, V = random_state(40, 24, 5, seed=19)
    assert step_violations(_mutant("none"), X, G, R, V, 0.01, 0.95, O.ORTH) == []


def test_golden_rank1_exact_case():
    """Hand-derived closed form stored in tests/golden/rank1_exact_3x2.json."""
    import json
    import os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "rank1_exact_3x2.json")))
    X, G, R, V = (np.array(fx[k], dtype=np.float64) for k in ("X", "G", "R", "V"))
    a = np.array([1.0, 2.0, 2.0])
    b = np.array([1.0, 2.0])
    U = a / 3.0
    Vb = b / math.sqrt(5.0)
    Xe = X - fx["eta"] * math.sqrt(3.0 / 2.0) * np.outer(U, Vb)
    for variant in (O.ORTH, O.DION):
        out = O.oracle_step(X, G, R, V, fx["eta"], fx["beta"], variant)
        assert np.abs(out["U"][:, 0] - U).max() < 1e-15
        assert np.abs(out["W"] - np.array(fx["expected"]["W"])).max() < 1e-14
        assert np.abs(out["Vbar"][:, 0] - Vb).max() < 1e-15
        assert np.abs(out["X"] - Xe).max() < 1e-15
        assert np.abs(out["R"]).max() < 1e-14
