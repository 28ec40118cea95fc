"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Every case draws seeded inputs (rank_orthonormalized_optimizer_03_b300.synth),
hands the same stored fp32 / bf16 values to both sides and compares
element-wise (relative Frobenius norms) with the tolerances of parity_util.
"""
import math

import numpy as np
import pytest

from oracle import dion_oracle as O
from parity_util import (TOL_CHAIN, TOL_ORTH, TOL_STEP, check_step, f64, grad_f64, grad_to_device,
                         orth_v0, padded, rel, state_snapshot)
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dion.lib()
    return torch.device("cuda:0")


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def host_matrix(hi, dev, variant):
    import torch
    s = hi.spec
    return dict(X=to_dev(hi.X0, dev), G=grad_to_device(hi.grads[0], dev),
                R=torch.zeros((s.m, s.n), dtype=torch.float32, device=dev),
                V=to_dev(orth_v0(hi.V0_raw), dev), eta=s.eta, beta=s.beta, variant=variant,
                scale=s.scale)


# ---------------------------------------------------------------- single matrices, chains
@pytest.mark.parametrize("variant", ["orth", "dion"])
@pytest.mark.parametrize("wname", ["single_256x128_r16", "square_1024_r256"])
def test_chain_single_matrix(dev, wname, variant):
    import torch
    wl = workloads.by_name(wname)
    hi = synth.host_inputs(wl, seed=0)
    s = hi.spec
    d = host_matrix(hi, dev, variant)
    plan = dion.Plan([d])
    # the oracle's own float64 trajectory from the same initial state
    traj = dict(X=f64(d["X"]), R=f64(d["R"]), V=f64(d["V"]))
    worst = {}
    for t in range(wl.steps):
        d["G"].copy_(grad_to_device(hi.grads[t], dev))
        before = state_snapshot(d)
        plan.step()
        torch.cuda.synchronize()
        assert plan.failures() == [0]
        G64 = hi.grad_f64(t)
        _, errs = check_step(before, G64, d, s.eta, s.beta, variant, s.scale,
                             U_gpu=plan.buffer(0, dion.BUF_U))
        for k, v in errs.items():
            worst[k] = max(worst.get(k, 0.0), v)
        ref = O.oracle_step(traj["X"], G64, traj["R"], traj["V"], s.eta, s.beta, variant, s.scale)
        traj = dict(X=ref["X"], R=ref["R"], V=ref["V"])
    after = state_snapshot(d)
    assert rel(after["X"], traj["X"]) <= TOL_CHAIN
    assert rel(after["R"], traj["R"]) <= TOL_CHAIN
    print(wname, variant, "worst single-step errors", worst)


# ---------------------------------------------------------------- batched models
def device_plan(wl, dev, variants=("orth",), indices=None, seed=0):
    mats = []
    for k, spec in enumerate(wl.mats):
        X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, k, seed=seed, device=dev)
        import torch
        V0 = to_dev(orth_v0(f64(V0_raw)), dev)
        mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=V0, eta=spec.eta, beta=spec.beta,
                         variant=variants[k % len(variants)], scale=spec.scale))
    return mats


def check_batched(wl, dev, check_idx, variants=("orth", "dion")):
    import torch
    mats = device_plan(wl, dev, variants)
    plan = dion.Plan(mats)
    before = {i: state_snapshot(mats[i]) for i in check_idx}
    G64 = {i: grad_f64(mats[i]["G"]) for i in check_idx}
    plan.step()
    torch.cuda.synchronize()
    st = plan.failures()
    assert all(v == 0 for v in st), st
    worst = {}
    for i in check_idx:
        spec = wl.mats[i]
        _, errs = check_step(before[i], G64[i], mats[i], spec.eta, spec.beta, mats[i]["variant"],
                             spec.scale, U_gpu=plan.buffer(i, dion.BUF_U))
        for k, v in errs.items():
            worst[k] = max(worst.get(k, 0.0), v)
    print(wl.name, "worst", worst)
    return plan, mats


def test_gpt160m_all_matrices(dev):
    wl = workloads.gpt_160m(4)
    check_batched(wl, dev, list(range(len(wl.mats))))


@pytest.mark.slow
@pytest.mark.parametrize("variant", ["orth", "dion"])
def test_gpt160m_chain_10_steps(dev, variant):
    """All 72 GPT-160M matrices stepped 10 times in one plan with fresh gradients
    every step (seeds 0..9).  Layers 0 and 11 (12 matrices) are checked every
    step from identical state (check_step) and, after 10 steps, against the
    oracle's own float64 trajectory from the same initial state (<= TOL_CHAIN)."""
    import torch
    wl = workloads.gpt_160m(4)
    mats = device_plan(wl, dev, (variant,))
    idx = list(range(0, 6)) + list(range(66, 72))
    plan = dion.Plan(mats)
    traj = {i: state_snapshot(mats[i]) for i in idx}
    worst = {}
    for t in range(10):
        if t > 0:
            for k, spec in enumerate(wl.mats):
                mats[k]["G"].copy_(synth.device_matrix_inputs(spec, wl, k, seed=t, device=dev)[2])
        torch.cuda.synchronize()
        before = {i: state_snapshot(mats[i]) for i in idx}
        G64 = {i: grad_f64(mats[i]["G"]) for i in idx}
        plan.step()
        torch.cuda.synchronize()
        assert plan.failures() == [0] * len(mats)
        for i in idx:
            spec = wl.mats[i]
            _, errs = check_step(before[i], G64[i], mats[i], spec.eta, spec.beta, variant, spec.scale,
                                 U_gpu=plan.buffer(i, dion.BUF_U), qr=O.lapack_qr_pos)
            for k, v in errs.items():
                worst[k] = max(worst.get(k, 0.0), v)
            ref = O.oracle_step(traj[i]["X"], G64[i], traj[i]["R"], traj[i]["V"], spec.eta, spec.beta, variant,
                                spec.scale, qr=O.lapack_qr_pos)
            traj[i] = dict(X=ref["X"], R=ref["R"], V=ref["V"])
    chain = {}
    for i in idx:
        after = state_snapshot(mats[i])
        chain[i] = (rel(after["X"], traj[i]["X"]), rel(after["R"], traj[i]["R"]))
        assert chain[i][0] <= TOL_CHAIN and chain[i][1] <= TOL_CHAIN, (wl.mats[i].name, chain[i])
    print(variant, "worst single-step", worst, "worst chain", max(max(v) for v in chain.values()))
    plan.close()


def ill_conditioned_case(m, n, r, eps, seed):
    """A step whose P = M V is ill conditioned through the warm start: M is an
    ordinary gradient (rank-4 signal A B^T plus noise), and V's first two columns
    lie in the noise subspace (orthogonal to B), nearly parallel: the second is
    the first plus eps times a unit vector.  For eps = 1e-2, kappa(P) ~ 1e4 and the
    smallest Cholesky pivot of P^T P is ~1e-7 of its largest diagonal entry (below
    1e-6: orth(P) takes the shifted branch).  The direction separating the two
    columns is eps of their size; an fp32-accurate product determines it to ~u/eps,
    which keeps the step within the tolerances here (at eps = 3e-4 the update is
    off by ~1e-2 on the GPU, as any fp32 computation of P would be).  (Nearly parallel columns in the signal subspace keep the pivot
    ratio near eps^2; an ill-conditioned M spectrum below its noise floor leaves
    W = M^T U ill determined in fp32 whatever the algorithm.)"""
    g = np.random.Generator(np.random.PCG64(seed))
    A, B = g.standard_normal((m, 4)), g.standard_normal((n, 4))
    G = A @ B.T + 0.1 * g.standard_normal((m, n))
    V, _ = np.linalg.qr(g.standard_normal((n, r)))
    Qb, _ = np.linalg.qr(B)
    for k in (0, 1):
        V[:, k] -= Qb @ (Qb.T @ V[:, k])
        V[:, k] /= np.linalg.norm(V[:, k])
    V[:, 1] = V[:, 0] + eps * V[:, 1]
    return G.astype(np.float32), V.astype(np.float32), g.normal(0, 0.02, (m, n)).astype(np.float32)


@pytest.mark.parametrize("variant", ["orth", "dion"])
def test_shifted_choleskyqr3_on_ill_conditioned_p(dev, variant):
    """kappa(P) ~ 1e4 is beyond fp32 CholeskyQR2 (kappa^2 u ~ 6): for Orth-Dion the
    first Cholesky's pivots must send orth(P) down the shifted CholeskyQR3 branch,
    which reports DION_MAT_SHIFTED and still returns the positive-diagonal Q factor;
    X, R, the update and Vbar against the oracle.  Dion first orthonormalises the
    warm start (orth(M V) = orth(M orth(V))), so its P is well conditioned and the
    step must match the oracle without the shifted branch; the branch on an
    orth(V)-like argument is covered by the no-alloc test's kappa ~ 1e4 case."""
    import torch
    m, n, r = 1024, 512, 32
    G, V, X = ill_conditioned_case(m, n, r, 1e-2, seed=31)
    d = dict(X=to_dev(X, dev), G=to_dev(G, dev), R=torch.zeros((m, n), device=dev), V=to_dev(V, dev),
             eta=0.02, beta=0.95, variant=variant)
    # a well-conditioned neighbour in the same plan must take the ordinary path
    g = np.random.Generator(np.random.PCG64(5))
    nb = dict(X=to_dev(g.normal(0, 0.02, (256, 128)), dev), G=to_dev(g.standard_normal((256, 128)), dev),
              R=torch.zeros((256, 128), device=dev), V=to_dev(orth_v0(g.standard_normal((128, 16))), dev),
              eta=0.02, beta=0.95, variant=variant)
    plan = dion.Plan([d, nb])
    before = [state_snapshot(d), state_snapshot(nb)]
    plan.step()
    torch.cuda.synchronize()
    st = plan.status()
    assert not st[0] & dion.FATAL, st
    if variant == "orth":
        assert st[0] & dion.DION_MAT_SHIFTED, st
    assert st[1] == 0, st
    ref, errs = check_step(before[0], f64(d["G"]), d, 0.02, 0.95, variant, U_gpu=plan.buffer(0, dion.BUF_U))
    from parity_util import kappa
    assert kappa(ref["P"]) > 5e3, kappa(ref["P"])
    check_step(before[1], f64(nb["G"]), nb, 0.02, 0.95, variant, U_gpu=plan.buffer(1, dion.BUF_U))
    print(variant, "kappa(P)", kappa(ref["P"]), "kappa(W)", kappa(ref["W"]), errs)
    plan.close()


@pytest.mark.slow
def test_llama3b_rdiv16_layers_0_and_27(dev):
    wl = workloads.llama_3b(16)
    idx = list(range(0, 7)) + list(range(27 * 7, 28 * 7))
    check_batched(wl, dev, idx)


# ---------------------------------------------------------------- per-phase intermediates
PHASE_CASES = [(100, 36, 1), (100, 36, 3), (36, 100, 17), (200, 64, 16), (64, 64, 64),
               (130, 260, 33), (257, 129, 2), (33, 48, 33)]


@pytest.mark.parametrize("m,n,r", PHASE_CASES)
@pytest.mark.parametrize("variant", ["orth", "dion"])
def test_phase_intermediates(dev, m, n, r, variant):
    import torch
    g = np.random.Generator(np.random.PCG64(m * 1000 + n * 10 + r))
    ld = ((n + 7) // 8) * 8 + 8           # padded row pitch, exercises ld > n
    X = padded(to_dev(g.normal(0, 0.02, (m, n)), dev), ld)
    R = padded(to_dev(0.05 * g.standard_normal((m, n)), dev), ld)
    Gn = (g.standard_normal((m, 4)) @ g.standard_normal((4, n)) + 0.1 * g.standard_normal((m, n)))
    G = padded(grad_to_device(synth.f32_to_bf16_bits(Gn.astype(np.float32)), dev), ld)
    V = to_dev(g.standard_normal((n, r)), dev)            # warm start need not be orthonormal
    d = dict(X=X, G=G, R=R, V=V, eta=0.03, beta=0.9, variant=variant)
    plan = dion.Plan([d])
    before = state_snapshot(d)
    G64 = grad_f64(G)
    ref = O.oracle_step(before["X"], G64, before["R"], before["V"], 0.03, 0.9, variant)
    plan.phases(0, 0)
    torch.cuda.synchronize()
    # Dion: phase (a) forms M orth(V), which has the same orth() as M V
    P_ref = ref["P"] if variant == "orth" else ref["M"] @ O.orth(before["V"])[0]
    assert rel(f64(plan.buffer(0, dion.BUF_P)), P_ref) < 1e-5
    plan.phases(1, 1)
    U = f64(plan.buffer(0, dion.BUF_U))
    assert np.abs(U.T @ U - np.eye(r)).max() < TOL_ORTH
    # The Q factor of a thin QR moves by up to kappa(P) times the relative
    # perturbation of P; P itself carries fp32 rounding (2^-24), so an
    # intermediate's forward error is bounded by a multiple of kappa(P) u,
    # not by a fixed number.  X and R below keep the fixed tolerances.
    sv = np.linalg.svd(P_ref, compute_uv=False)
    tol_mid = max(1e-4, 4.0 * (sv[0] / sv[-1]) * 2.0 ** -24)
    assert rel(U, ref["U"]) < tol_mid
    plan.phases(2, 2)
    assert rel(f64(plan.buffer(0, dion.BUF_W)), ref["W"]) < tol_mid
    plan.phases(3, 3)
    assert rel(f64(d["V"]), ref["Vbar"]) < tol_mid
    plan.phases(4, 4)
    torch.cuda.synchronize()
    assert plan.failures() == [0]
    assert rel(f64(d["X"]), ref["X"]) < TOL_STEP
    if r == min(m, n):
        # full rank: U U^T M = M, the residual vanishes; only fp32 rounding residue is left
        assert np.linalg.norm(f64(d["R"])) <= 1e-5 * 0.9 * np.linalg.norm(ref["M"])
    else:
        assert rel(f64(d["R"]), ref["R"]) < TOL_STEP
    assert rel(f64(d["X"]) - before["X"], ref["X"] - before["X"]) < 1e-3


def test_mixed_batch_dtypes_variants_shapes(dev):
    import torch
    g = np.random.Generator(np.random.PCG64(7))
    mats, refs, befores = [], [], []
    for k, (m, n, r, gdt, var) in enumerate([(96, 64, 8, "f32", "orth"), (64, 96, 8, "bf16", "dion"),
                                             (128, 128, 32, "bf16", "orth"), (48, 40, 1, "f32", "dion")]):
        X = to_dev(g.normal(0, 0.02, (m, n)), dev)
        R = to_dev(0.02 * g.standard_normal((m, n)), dev)
        Gn = (g.standard_normal((m, n)) * 0.1 + g.standard_normal((m, 2)) @ g.standard_normal((2, n)))
        G = grad_to_device(synth.f32_to_bf16_bits(Gn.astype(np.float32)) if gdt == "bf16"
                           else Gn.astype(np.float32), dev)
        V = to_dev(orth_v0(g.standard_normal((n, r))), dev)
        d = dict(X=X, G=G, R=R, V=V, eta=0.01 * (k + 1), beta=0.9, variant=var, scale=1.5 if k == 2 else 0.0)
        mats.append(d)
    plan = dion.Plan(mats)
    befores = [state_snapshot(d) for d in mats]
    plan.step()
    torch.cuda.synchronize()
    assert plan.failures() == [0, 0, 0, 0]
    for k, d in enumerate(mats):
        sc = 1.5 if k == 2 else None
        check_step(befores[k], grad_f64(d["G"]), d, d["eta"], d["beta"], d["variant"], sc,
                   U_gpu=plan.buffer(k, dion.BUF_U))


def test_update_in_k_passes_mixed_ranks(dev):
    """Ranks above 256 take the update in several K passes (at most 256 of K
    accumulated on the tensor core per launch); a batch mixing one, two and
    three passes against the oracle."""
    import torch
    g = np.random.Generator(np.random.PCG64(11))
    # bf16 row pitches stay multiples of 16 bytes (n a multiple of 8)
    shapes = [(200, 160, 16, "orth"), (700, 600, 400, "orth"), (520, 896, 300, "dion"), (1100, 640, 520, "orth")]
    mats = []
    for m, n, r, var in shapes:
        X = to_dev(g.normal(0, 0.02, (m, n)), dev)
        R = to_dev(0.05 * g.standard_normal((m, n)), dev)
        Gn = g.standard_normal((m, n)) + 0.2 * (g.standard_normal((m, 2)) @ g.standard_normal((2, n)))
        G = grad_to_device(synth.f32_to_bf16_bits(Gn.astype(np.float32)), dev)
        V = to_dev(g.standard_normal((n, r)) / math.sqrt(n), dev)
        mats.append(dict(X=X, G=G, R=R, V=V, eta=0.02, beta=0.95, variant=var))
    plan = dion.Plan(mats)
    assert plan.launches_per_step > 0
    befores = [state_snapshot(d) for d in mats]
    plan.step()
    torch.cuda.synchronize()
    assert plan.failures() == [0] * len(mats)
    for k, d in enumerate(mats):
        _, errs = check_step(befores[k], grad_f64(d["G"]), d, 0.02, 0.95, d["variant"],
                             U_gpu=plan.buffer(k, dion.BUF_U))
        print(shapes[k], errs)


# ---------------------------------------------------------------- failure handling
def test_rank_deficient_sets_status_and_leaves_state(dev):
    import torch
    m, n, r = 64, 32, 4
    X = torch.randn(m, n, device=dev)
    R = torch.zeros(m, n, device=dev)
    G = torch.zeros(m, n, device=dev)
    V = torch.randn(n, r, device=dev)
    ok = dict(X=torch.randn(m, n, device=dev), G=torch.randn(m, n, device=dev), R=torch.zeros(m, n, device=dev),
              V=torch.randn(n, r, device=dev), eta=0.1, beta=0.9)
    snap = [t.clone() for t in (X, R, V)]
    plan = dion.Plan([dict(X=X, G=G, R=R, V=V, eta=0.1, beta=0.9), ok])
    plan.step()
    torch.cuda.synchronize()
    st = plan.status()
    assert st[0] & dion.DION_MAT_CHOL_BREAKDOWN and (st[1] & dion.FATAL) == 0
    for a, b in zip((X, R, V), snap):
        assert torch.equal(a, b)


def test_nonfinite_gradient_sets_status(dev):
    import torch
    m, n, r = 64, 32, 4
    G = torch.randn(m, n, device=dev)
    G[3, 5] = float("nan")
    X = torch.randn(m, n, device=dev)
    R = torch.zeros(m, n, device=dev)
    V = torch.randn(n, r, device=dev)
    snap = [t.clone() for t in (X, R, V)]
    plan = dion.Plan([dict(X=X, G=G, R=R, V=V, eta=0.1, beta=0.9)])
    plan.step()
    torch.cuda.synchronize()
    st = plan.status()
    assert st[0] & dion.DION_MAT_NONFINITE
    for a, b in zip((X, R, V), snap):
        assert torch.equal(a, b)


# ---------------------------------------------------------------- determinism, resume
def test_bitwise_deterministic_and_resumable(dev):
    import torch
    wl = workloads.gpt_160m(4)
    sub = workloads.Workload("gpt_sub", wl.mats[:6], wl.g_dtype, wl.grad, wl.grad_rank, wl.grad_noise,
                             wl.grad_signal)
    a = device_plan(sub, dev, ("orth", "dion"))
    b = [{k: (v.clone() if hasattr(v, "clone") else v) for k, v in d.items()} for d in a]
    pa, pb = dion.Plan(a), dion.Plan(b)
    for _ in range(3):
        pa.step()
        pb.step()
    torch.cuda.synchronize()
    for da, db in zip(a, b):
        for k in ("X", "R", "V"):
            assert torch.equal(da[k], db[k])
    # checkpoint after 3 steps, resume with a fresh plan on the saved state, 2 more steps
    c = [{k: (v.clone() if hasattr(v, "clone") else v) for k, v in d.items()} for d in a]
    for _ in range(2):
        pa.step()
    pc = dion.Plan(c)
    for _ in range(2):
        pc.step()
    torch.cuda.synchronize()
    for da, dc in zip(a, c):
        for k in ("X", "R", "V"):
            assert torch.equal(da[k], dc[k])


def test_set_hparams_takes_effect(dev):
    import torch
    g = np.random.Generator(np.random.PCG64(3))
    m, n, r = 64, 48, 4
    d = dict(X=to_dev(g.normal(0, 0.02, (m, n)), dev), G=to_dev(g.standard_normal((m, n)), dev),
             R=torch.zeros(m, n, device=dev), V=to_dev(orth_v0(g.standard_normal((n, r))), dev),
             eta=0.01, beta=0.9)
    plan = dion.Plan([d])
    plan.set_hparams(0, 0.2, 0.5)
    before = state_snapshot(d)
    plan.step()
    torch.cuda.synchronize()
    check_step(before, grad_f64(d["G"]), d, 0.2, 0.5, "orth")


@pytest.mark.parametrize("variant", ["dion", "orth"])
def test_consecutive_steps_from_random_warm_start(dev, variant):
    """Step 2 of Dion starts from Vbar = colnorm(W), whose condition number is ~2e2 here;
    with a strong low-rank gradient M Vbar then has condition ~1e4, beyond fp32 CholeskyQR.
    The step must still match the oracle (the library orthonormalises V first)."""
    import torch
    wl = workloads.gpt_160m(4)
    spec = wl.mats[4]                                   # 3072 x 768, r = 192
    X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, 4, seed=1, device=dev)
    d = dict(X=X0, G=G, R=torch.zeros_like(X0), V=to_dev(orth_v0(f64(V0_raw)), dev), eta=spec.eta,
             beta=spec.beta, variant=variant, scale=spec.scale)
    plan = dion.Plan([d])
    G64 = grad_f64(G)
    for _ in range(3):
        before = state_snapshot(d)
        plan.step()
        torch.cuda.synchronize()
        assert plan.failures() == [0]
        check_step(before, G64, d, spec.eta, spec.beta, variant, spec.scale, U_gpu=plan.buffer(0, dion.BUF_U))
