"""dion_orth_noalloc: orth() for callers that cannot allocate device memory.

Callers inside a CUDA graph capture, an allocator callback, or a framework
that owns every device byte cannot give the library a workspace.  This entry
point keeps its scratch in a fixed array inside libdion.so.  The test calls it
through the C ABI twice in a row, each time on the P of a plan-based step, and
checks the result against the U = orth(P) that the plan-based entry point
produced from the same P and against the oracle's Householder Q factor, with
the tolerances of the other parity tests.  An ill-conditioned argument
(kappa ~ 1e4) must take the shifted CholeskyQR3 branch through the same fixed
scratch.  A request beyond the fixed scratch is refused cleanly.  The file is
collected last so that a failure here cannot hide the other tests.
"""
import numpy as np
import pytest

from oracle import dion_oracle as O
from parity_util import TOL_ORTH, f64, grad_to_device, rel
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dion.lib()
    return torch.device("cuda:0")


def plan_orth_of_p(dev, m, n, r, seed):
    """P = (G + R) V and U = orth(P) from the plan-based step (phases a and b)."""
    import torch
    g = np.random.Generator(np.random.PCG64(seed))
    X = torch.from_numpy(g.normal(0, 0.02, (m, n)).astype(np.float32)).to(dev)
    R = torch.from_numpy((0.05 * g.standard_normal((m, n))).astype(np.float32)).to(dev)
    Gn = g.standard_normal((m, 4)) @ g.standard_normal((4, n)) + 0.1 * g.standard_normal((m, n))
    G = grad_to_device(synth.f32_to_bf16_bits(Gn.astype(np.float32)), dev)
    V = torch.from_numpy(np.linalg.qr(g.standard_normal((n, r)))[0].astype(np.float32)).to(dev)
    plan = dion.Plan([dict(X=X, G=G, R=R, V=V, eta=0.02, beta=0.95, variant="orth")])
    plan.phases(0, 1)
    torch.cuda.synchronize()
    assert plan.failures() == [0]
    return plan, plan.buffer(0, dion.BUF_P), plan.buffer(0, dion.BUF_U)


def test_orth_noalloc_matches_plan_orth_on_two_calls(dev):
    import torch
    for m, n, r, seed in [(1000, 296, 48, 11), (2048, 512, 64, 12)]:
        plan, P, U = plan_orth_of_p(dev, m, n, r, seed)
        Q = torch.full((m, r), float("nan"), dtype=torch.float32, device=dev)
        st = dion.orth_noalloc(P, Q)
        assert st & dion.FATAL == 0, st
        Qh, Uh, Ph = f64(Q), f64(U), f64(P)
        sv = np.linalg.svd(Ph, compute_uv=False)
        tol = max(1e-4, 4.0 * (sv[0] / sv[-1]) * 2.0 ** -24)
        assert rel(Qh, Uh) < tol
        assert rel(Qh, O.householder_qr_pos(Ph)[0]) < tol
        assert np.abs(Qh.T @ Qh - np.eye(r)).max() < TOL_ORTH
        plan.close()


def test_orth_noalloc_ill_conditioned_takes_shifted_path(dev):
    """kappa(A) ~ 1e4: the first Cholesky's pivots send the call down shifted
    CholeskyQR3 (status DION_MAT_SHIFTED), whose second factor Q2 also lives in
    the fixed scratch; Q still equals the oracle's positive-diagonal Q factor."""
    import torch
    rows, r = 1000, 48
    g = np.random.Generator(np.random.PCG64(41))
    Qa, _ = np.linalg.qr(g.standard_normal((rows, r)))
    Z, _ = np.linalg.qr(g.standard_normal((r, r)))
    A = ((Qa * np.geomspace(1.0, 1e-4, r)[None, :]) @ Z.T).astype(np.float32)
    Ad = torch.from_numpy(A).to(dev)
    Ah = A.astype(np.float64)
    ref = O.householder_qr_pos(Ah)[0]
    sv = np.linalg.svd(Ah, compute_uv=False)
    assert sv[0] / sv[-1] > 5e3
    tol = max(1e-4, 4.0 * (sv[0] / sv[-1]) * 2.0 ** -24)
    for _ in range(2):
        Q = torch.full((rows, r), float("nan"), dtype=torch.float32, device=dev)
        st = dion.orth_noalloc(Ad, Q)
        assert st & dion.DION_MAT_SHIFTED and not st & dion.FATAL, st
        Qh = f64(Q)
        assert np.abs(Qh.T @ Qh - np.eye(r)).max() < TOL_ORTH
        assert rel(Qh, ref) < tol


def test_orth_noalloc_refuses_sizes_beyond_its_scratch(dev):
    import torch
    A = torch.zeros((dion.NOALLOC_MAX_ROWS + 1, 8), dtype=torch.float32, device=dev)
    with pytest.raises(dion.DionError) as e:
        dion.orth_noalloc(A, torch.empty_like(A))
    assert e.value.code == dion.DION_ERR_UNSUPPORTED
    B = torch.zeros((128, dion.NOALLOC_MAX_RANK + 1), dtype=torch.float32, device=dev)
    with pytest.raises(dion.DionError) as e:
        dion.orth_noalloc(B, torch.empty_like(B))
    assert e.value.code == dion.DION_ERR_UNSUPPORTED
