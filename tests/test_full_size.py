"""GPU parity at full workload sizes: the single-matrix rank sweep (8192 x 8192
and 4096 x 16384, r = 32 ... 2048) and the Llama-3B shapes at rank min(m, n)/4.

Where the float64 oracle finishes in seconds (small r, sampled matrices of a
batch) the whole step is compared with it.  Elsewhere the step is checked
against properties that define each factor at any size, computed in float64
on the host from the stored inputs and the GPU's own factors:

* U = orth(M V): U^T U = I, and C = U^T (M V) is upper triangular with a
  positive diagonal and reproduces M V = U C.  An orthonormal U with that
  property is the Q factor of the thin QR of M V (unique for a full-rank
  argument), which is the glossary's orth() under the positive-diagonal
  reading.
* W = M^T U, to the accuracy of one fp32 contraction.
* Vbar: the same QR characterisation for W (Orth-Dion), or W's columns scaled
  to unit length (Dion).
* X' = X - eta s U Vbar^T and R' = beta (M - U W^T) from those factors.

P, W, X' and R' are compared on one sampled row (column) in every tile of
128, so that every tile of every launch is looked at.

junaidaliop.github.io "Orth-Dion", the update equations and the symbol
glossary under them.
"""
import math

import numpy as np
import pytest

from oracle import dion_oracle as O
from parity_util import TOL_ORTH, TOL_STEP, check_step, f64, grad_f64, rel, state_snapshot
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth, workloads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_GEMM = 3e-5      # one fp32-accurate (3xTF32) contraction against float64


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dion.lib()
    return torch.device("cuda:0")


def qr_tolerance(A):
    """Forward-error budget of the Q factor of A: the relative perturbation of A
    (fp32 storage, 2^-24) amplified by kappa(A), never below the step tolerance."""
    ev = np.linalg.eigvalsh(A.T @ A)
    kappa = math.sqrt(ev[-1] / max(ev[0], 1e-300))
    return max(TOL_STEP, 4.0 * kappa * 2.0 ** -24), kappa


def assert_is_q_factor(Q, A, what):
    """Q (rows x r) is the thin-QR Q factor of A with a positive-diagonal R."""
    r = A.shape[1]
    assert np.abs(Q.T @ Q - np.eye(r)).max() <= TOL_ORTH, what + ": not orthonormal"
    tol, kappa = qr_tolerance(A)
    C = Q.T @ A
    assert rel(Q @ C, A) <= tol, (what, "span", rel(Q @ C, A), kappa)
    low = np.linalg.norm(np.tril(C, -1)) / np.linalg.norm(C)
    assert low <= tol, (what, "triangular", low, kappa)
    assert (np.diag(C) > 0).all(), what + ": diagonal of Q^T A not positive"


def strata(extent, tile, gen):
    """One random index inside every tile of ``tile`` along an axis of ``extent``."""
    return np.array([t + int(gen.integers(0, min(tile, extent - t))) for t in range(0, extent, tile)])


def snapshot_samples(d, rows, cols):
    """Float64 host copies of what the property checks read before the step:
    the sampled rows and columns of X, G and R, and V."""
    import torch
    ri = torch.as_tensor(rows, device=d["X"].device)
    ci = torch.as_tensor(cols, device=d["X"].device)
    return {"X_rows": f64(d["X"][ri]), "M_rows": f64(d["G"][ri]) + f64(d["R"][ri]),
            "M_cols": f64(d["G"][:, ci]) + f64(d["R"][:, ci]), "V": f64(d["V"])}


def check_updates(snap, d, rows, U, W, Vbar, eta, beta, scale):
    """X' = X - eta s U Vbar^T and R' = beta (M - U W^T) on the sampled rows."""
    import torch
    ri = torch.as_tensor(rows, device=d["X"].device)
    X1, R1 = f64(d["X"][ri]), f64(d["R"][ri])
    X_ref = snap["X_rows"] - eta * scale * (U[rows] @ Vbar.T)
    R_ref = beta * (snap["M_rows"] - U[rows] @ W.T)
    errs = {"X": rel(X1, X_ref), "dX": rel(X1 - snap["X_rows"], X_ref - snap["X_rows"]), "R": rel(R1, R_ref)}
    assert errs["X"] <= TOL_STEP and errs["R"] <= TOL_STEP and errs["dX"] <= 1e-3, errs
    return errs


def sweep_case(shape, r, variants):
    """One step of an Orth-Dion matrix (and, when asked, a Dion matrix with the
    same inputs) in one plan; r = 32 against the oracle, larger r by properties."""
    import torch
    devc = torch.device("cuda:0")
    wl = workloads.sweep(shape, r)
    spec = wl.mats[0]
    mats = []
    for v in variants:
        X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, 0, seed=0, device=devc)
        V0 = (V0_raw / math.sqrt(spec.n)).contiguous()
        mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=V0, eta=spec.eta, beta=spec.beta, variant=v,
                         scale=spec.scale))
    scale = spec.scale if spec.scale else math.sqrt(spec.m / spec.n)
    gen = np.random.Generator(np.random.PCG64(r))
    rows, cols = strata(spec.m, 128, gen), strata(spec.n, 128, gen)
    # element-wise against the oracle at the ends and the middle of the sweep
    # (LAPACK's QR inside the oracle above r = 32: its textbook loop takes minutes there)
    oracle = r in (32, 256, 2048)
    if oracle:
        before = [state_snapshot(d) for d in mats]
        G64 = grad_f64(mats[0]["G"])
    else:
        snaps = [snapshot_samples(d, rows, cols) for d in mats]
    plan = dion.Plan(mats)
    plan.step()
    torch.cuda.synchronize()
    assert plan.failures() == [0] * len(mats)
    out = []
    if oracle:
        for k, v in enumerate(variants):
            _, errs = check_step(before[k], G64, mats[k], spec.eta, spec.beta, v, spec.scale,
                                 U_gpu=plan.buffer(k, dion.BUF_U), qr=None if r <= 32 else O.lapack_qr_pos)
            out.append((v, errs))
        plan.close()
        return out
    # Orth-Dion matrix (index 0): every factor by its defining property
    s0 = snaps[0]
    P = f64(plan.buffer(0, dion.BUF_P))
    U = f64(plan.buffer(0, dion.BUF_U))
    W = f64(plan.buffer(0, dion.BUF_W))
    Vbar = f64(mats[0]["V"])
    errs = {"P": rel(P[rows], s0["M_rows"] @ s0["V"])}
    assert errs["P"] <= TOL_GEMM, errs
    assert_is_q_factor(U, P, "U")
    errs["W"] = rel(W[cols], s0["M_cols"].T @ U)
    assert errs["W"] <= TOL_GEMM, errs
    assert_is_q_factor(Vbar, W, "Vbar")
    errs.update(check_updates(s0, mats[0], rows, U, W, Vbar, spec.eta, spec.beta, scale))
    out.append(("orth", errs))
    if len(variants) > 1:
        # Dion matrix (index 1), same inputs: U and W equal the Orth-Dion ones
        # (orth(M V) does not depend on which basis of span(V) phase (a) reads);
        # Vbar is W with unit columns
        s1 = snaps[1]
        tol, _ = qr_tolerance(P)
        Ud = f64(plan.buffer(1, dion.BUF_U))
        Wd = f64(plan.buffer(1, dion.BUF_W))
        Vd = f64(mats[1]["V"])
        e = {"U": rel(Ud, U), "W": rel(Wd[cols], s1["M_cols"].T @ Ud)}
        assert e["U"] <= tol and e["W"] <= TOL_GEMM, e
        e["Vbar"] = rel(Vd, Wd / np.linalg.norm(Wd, axis=0))
        assert e["Vbar"] <= TOL_GEMM, e
        e.update(check_updates(s1, mats[1], rows, Ud, Wd, Vd, spec.eta, spec.beta, scale))
        out.append(("dion", e))
    plan.close()
    return out


@pytest.mark.parametrize("r", workloads.SWEEP_RANKS)
@pytest.mark.parametrize("shape", workloads.SWEEP_SHAPES)
def test_rank_sweep(dev, shape, r):
    variants = ("orth", "dion") if r in (32, 256, 2048) else ("orth",)
    for v, errs in sweep_case(shape, r, variants):
        print(shape, r, v, errs)


def test_llama3b_rdiv4_sampled_matrices(dev):
    """All 196 matrices at r = min(m, n)/4 (768, or 256 for k and v) in one plan,
    as the step runs; the oracle checks the whole of layer 0 (seven matrices,
    both variants, r = 256 and 768) and layer 27's k (Dion, r = 256)."""
    import torch
    wl = workloads.llama_3b(4)
    mats = []
    for k, spec in enumerate(wl.mats):
        X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, k, seed=0, device=dev)
        # the raw Gaussian warm start scaled by 1/sqrt(n), as the benchmark steps it
        mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=(V0_raw / math.sqrt(spec.n)).contiguous(),
                         eta=spec.eta, beta=spec.beta, variant=("orth", "dion")[k % 2], scale=spec.scale))
    idx = list(range(7)) + [27 * 7 + 1]
    before = {i: state_snapshot(mats[i]) for i in idx}
    G64 = {i: grad_f64(mats[i]["G"]) for i in idx}
    plan = dion.Plan(mats)
    plan.step()
    torch.cuda.synchronize()
    st = plan.failures()
    assert all(v == 0 for v in st), st
    for i in idx:
        spec = wl.mats[i]
        _, errs = check_step(before[i], G64[i], mats[i], spec.eta, spec.beta, mats[i]["variant"], spec.scale,
                             U_gpu=plan.buffer(i, dion.BUF_U), qr=O.lapack_qr_pos)
        print(spec.name, mats[i]["variant"], errs)
    plan.close()
