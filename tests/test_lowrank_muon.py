"""Low-rank Muon variant (DION_VARIANT_LOWRANK_MUON): its float64 oracle's pins
on the CPU, and the library's step against that oracle on the GPU.

The algorithm is this library's reading (the pages give none), so parity is
unpinned beyond the reading; the pins check that the oracle computes what the
reading states: the momentum closed form, the update's singular values and
spaces on an exact-rank momentum, agreement with the (pinned) Orth-Dion
oracle step on M = G + mu B, and planted slips.
"""
import math

import numpy as np
import pytest

from oracle import dion_oracle as O
from oracle.lowrank_muon_oracle import lowrank_muon_step
from parity_util import TOL_DX, TOL_STEP, f64, grad_to_device, rel
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def test_momentum_closed_form():
    g = rng(1)
    G = g.standard_normal((20, 12))
    B = np.zeros((20, 12))
    for t in range(1, 5):
        B = lowrank_muon_step(np.zeros((20, 12)), G, B, g.standard_normal((12, 3)), 0.1, 0.9)["B"]
        assert np.abs(B - G * (1 - 0.9 ** t) / (1 - 0.9)).max() < 1e-13


def test_exact_rank_update_is_a_partial_isometry_on_the_momentum():
    """M of exact rank r: U Vbar^T has r unit singular values, column space col(M), row space row(M)."""
    g = rng(2)
    m, n, r = 30, 20, 4
    A, Bm = g.standard_normal((m, r)), g.standard_normal((n, r))
    M = A @ Bm.T
    out = lowrank_muon_step(np.zeros((m, n)), M, np.zeros((m, n)), g.standard_normal((n, r)), 1.0, 0.5, scale=1.0)
    D = -out["X"]
    sv = np.linalg.svd(D, compute_uv=False)
    assert np.abs(sv[:r] - 1).max() < 1e-12 and np.abs(sv[r:]).max() < 1e-12
    Qa = np.linalg.qr(A)[0]
    Qb = np.linalg.qr(Bm)[0]
    assert np.abs(D - Qa @ (Qa.T @ D)).max() < 1e-12
    assert np.abs(D - (D @ Qb) @ Qb.T).max() < 1e-12


def test_agrees_with_the_orth_dion_oracle_on_the_momentum():
    g = rng(3)
    m, n, r = 40, 25, 5
    X, G, B, Om = (g.standard_normal(s) for s in ((m, n), (m, n), (m, n), (n, r)))
    a = lowrank_muon_step(X, G, B, Om, 0.02, 0.9)
    b = O.oracle_step(X, G + 0.9 * B, np.zeros((m, n)), Om, 0.02, 0.0, O.ORTH)
    for k in ("X", "U", "W", "Vbar"):
        assert np.abs(a[k] - b[k]).max() < 1e-12, k


def _mutant(kind):
    def step(X, G, B, Om, eta, mu, scale=None):
        out = lowrank_muon_step(X, G, B, Om, eta, mu, scale)
        if kind == "error_feedback":
            out["B"] = out["B"] - out["U"] @ out["W"].T
        elif kind == "momentum_swapped":
            out["B"] = B + mu * G
        return out
    return step


@pytest.mark.parametrize("kind", ["error_feedback", "momentum_swapped"])
def test_planted_slips_fail_the_momentum_pin(kind):
    g = rng(4)
    G = g.standard_normal((20, 12))
    B = np.zeros((20, 12))
    bad = False
    for t in range(1, 4):
        B = _mutant(kind)(np.zeros((20, 12)), G, B, g.standard_normal((12, 3)), 0.1, 0.9)["B"]
        bad |= np.abs(B - G * (1 - 0.9 ** t) / (1 - 0.9)).max() > 1e-9
    assert bad


@pytest.mark.gpu
def test_lowrank_muon_steps_against_oracle():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dev = torch.device("cuda:0")
    g = rng(5)
    shapes = [(1024, 768, 32), (768, 1024, 64), (512, 512, 300)]
    mats = []
    for m, n, r in shapes:
        X = torch.from_numpy(g.normal(0, 0.02, (m, n)).astype(np.float32)).to(dev)
        mats.append(dict(X=X, G=torch.zeros((m, n), dtype=torch.bfloat16, device=dev),
                         R=torch.zeros((m, n), device=dev), V=torch.zeros((n, r), device=dev),
                         eta=0.02, beta=0.9, variant="lowrank_muon"))
    plan = dion.Plan(mats)
    gen = torch.Generator(device=dev)
    for t in range(2):
        for d, (m, n, r) in zip(mats, shapes):
            Gn = g.standard_normal((m, 3)) @ g.standard_normal((3, n)) + 0.1 * g.standard_normal((m, n))
            d["G"].copy_(grad_to_device(synth.f32_to_bf16_bits(Gn.astype(np.float32)), dev))
            gen.manual_seed(1000 * t + r)
            d["V"].copy_(torch.randn((n, r), generator=gen, device=dev) / math.sqrt(n))   # the fresh sketch
        before = [(f64(d["X"]), f64(d["G"]), f64(d["R"]), f64(d["V"])) for d in mats]
        plan.step()
        torch.cuda.synchronize()
        assert plan.failures() == [0] * len(mats)
        for d, (X0, G0, B0, Om) in zip(mats, before):
            ref = lowrank_muon_step(X0, G0, B0, Om, 0.02, 0.9, qr=O.lapack_qr_pos)
            e = {"X": rel(f64(d["X"]), ref["X"]), "dX": rel(f64(d["X"]) - X0, ref["X"] - X0),
                 "B": rel(f64(d["R"]), ref["B"])}
            assert e["X"] <= TOL_STEP and e["dX"] <= TOL_DX and e["B"] <= 1e-6, (d["X"].shape, t, e)
    plan.close()
