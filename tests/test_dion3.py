"""Dion3 row-selection variant (muon plan with row_fraction < 1): its float64
oracle's pins on the CPU, and the library's step against it on the GPU.

The selection rule is this library's reading (parity unpinned beyond it); the
pins check the oracle against what the reading states: the top-k rows by an
independent sort, the untouched rows, the singular-value map of the update
on the selected block (numpy SVD), Muon itself at row_fraction = 1, and
planted slips.  On the GPU the selected set is checked for validity (no
unselected row longer than a selected one, to fp32 rounding of the norms) and
the oracle then follows the GPU's selection.
"""
import math

import numpy as np
import pytest

from oracle import muon_oracle as MU
from oracle.dion3_oracle import dion3_step, select_rows
from parity_util import f64, grad_to_device, rel
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def pins(step, seed=0):
    g = rng(seed)
    m, n, rho, it = 40, 16, 0.3, 4
    X, G, B = g.standard_normal((m, n)), g.standard_normal((m, n)), g.standard_normal((m, n))
    out = step(X, G, B, 0.1, 0.9, it, rho, 1.2)
    Bn = 0.9 * B + G
    k = math.ceil(rho * m)
    norms = np.sum(Bn ** 2, axis=1)
    top = np.sort(np.argsort(-norms, kind="stable")[:k])
    bad = []
    if not np.array_equal(np.asarray(out["selected"]), top):
        bad.append("selection")
    rest = np.setdiff1d(np.arange(m), top)
    if np.abs(out["X"][rest] - X[rest]).max() != 0.0:
        bad.append("unselected rows changed")
    U, sv, Vt = np.linalg.svd(Bn[top], full_matrices=False)
    sv = sv / math.sqrt(np.sum(sv ** 2))
    for _ in range(it):
        sv = 1.5 * sv - 0.5 * sv ** 3
    if np.abs(out["X"][top] - (X[top] - 0.1 * 1.2 * (U * sv[None, :]) @ Vt)).max() > 1e-12:
        bad.append("update of the selected block")
    return bad


def test_oracle_pins():
    assert pins(dion3_step) == []


def test_full_fraction_is_muon():
    g = rng(1)
    X, G, B = g.standard_normal((12, 9)), g.standard_normal((12, 9)), g.standard_normal((12, 9))
    a = dion3_step(X, G, B, 0.1, 0.9, 5, 1.0)
    b = MU.muon_step(X, G, B, 0.1, 0.9, 5)
    assert np.abs(a["X"] - b["X"]).max() < 1e-14


def test_ties_go_to_the_lower_row():
    B = np.ones((6, 3))
    assert list(select_rows(B, 2)) == [0, 1]


def _mutant(kind):
    def step(X, G, B, eta, mu, it, rho, scale=None):
        X = np.array(X, dtype=np.float64)
        Bn = mu * B + G
        m = X.shape[0]
        k = math.ceil(rho * m)
        norms = np.sum(Bn ** 2, axis=1)
        S = np.sort(np.argsort(norms if kind == "smallest" else -norms, kind="stable")[:k])
        Y0 = Bn[S] / (np.linalg.norm(Bn) if kind == "whole_norm" else np.linalg.norm(Bn[S]))
        Y = Y0
        for _ in range(it):
            Y = 1.5 * Y - 0.5 * ((Y @ Y.T) @ Y)
        if kind == "all_rows":
            X -= eta * scale * MU.ns_cubic(Bn, it)
        else:
            X[S] -= eta * scale * Y
        return {"X": X, "B": Bn, "selected": S}
    return step


@pytest.mark.parametrize("kind", ["smallest", "whole_norm", "all_rows"])
def test_planted_slips_are_caught(kind):
    assert pins(_mutant(kind)), kind
    assert pins(_mutant("none")) == []


@pytest.mark.gpu
@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_row_selection_against_oracle(precision):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dev = torch.device("cuda:0")
    g = rng(7)
    shapes = [(300, 128), (768, 3072), (3072, 768), (100, 40)]
    iters, rho = 5, 0.25
    mats = []
    for m, n in shapes:
        mats.append(dict(X=torch.from_numpy(g.normal(0, 0.02, (m, n)).astype(np.float32)).to(dev),
                         G=torch.zeros((m, n), dtype=torch.bfloat16, device=dev), B=torch.zeros((m, n), device=dev),
                         eta=0.02, mu=0.95))
    plan = dion.MuonPlan(mats, iters=iters, precision=precision, row_fraction=rho)
    for t in range(2):
        for d, (m, n) in zip(mats, shapes):
            Gn = (g.standard_normal((m, n)) * np.exp(g.standard_normal((m, 1)))).astype(np.float32)
            d["G"].copy_(grad_to_device(synth.f32_to_bf16_bits(Gn), dev))
        before = [(f64(d["X"]), f64(d["G"]), f64(d["B"])) for d in mats]
        plan.step()
        torch.cuda.synchronize()
        for i, (d, (X0, G0, B0)) in enumerate(zip(mats, before)):
            m, n = d["X"].shape
            sel = plan.selected_rows(i).cpu().numpy().astype(np.int64)
            k = math.ceil(rho * m)
            assert len(sel) == k and np.all(np.diff(sel) > 0)
            Bg = f64(d["B"])
            norms = np.sum(Bg ** 2, axis=1)
            rest = np.setdiff1d(np.arange(m), sel)
            # valid: no unselected row longer than a selected one (fp32 sums of n squares)
            assert norms[rest].max() <= norms[sel].min() * (1 + 4 * n * 2.0 ** -24)
            ref = dion3_step(X0, G0, B0, 0.02, 0.95, iters, rho, selected=sel)
            Xg = f64(d["X"])
            assert np.array_equal(Xg[rest], X0[rest])                  # untouched rows, bitwise
            e = {"dX": rel(Xg[sel] - X0[sel], ref["X"][sel] - X0[sel]), "B": rel(Bg, ref["B"])}
            amp = 1.5 ** iters
            tol = amp * (4 * math.sqrt(n) * 2.0 ** -24 if precision == "fp32" else 4 * 2.0 ** -8)
            assert e["B"] <= 1e-6 and e["dX"] <= max(tol, 1e-6), (m, n, t, e, tol)
    plan.close()
