"""GPU parity of the Muon comparator (include/muon.h) against its float64 oracle.

Two chained steps (the momentum carries over) of a batch mixing shapes with
m < n, m = n and m > n and both gradient dtypes, in each precision mode of
the Newton-Schulz products.  The bound on the update Y_K is derived from the
arithmetic: every iteration maps a singular value s to 1.5 s - 0.5 s^3, whose
slope is at most 1.5, so a relative error e made in one product grows by at
most 1.5 per later iteration; with K iterations and products accurate to e
(fp32: 4 sqrt(k) 2^-24 for an inner dimension k; tf32 operands: 4 * 2^-11;
bf16 storage: 4 * 2^-8) the bound is 1.5^K e.
"""
import math

import numpy as np
import pytest

from oracle import muon_oracle as MU
from parity_util import f64, grad_to_device, rel
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


SHAPES = [(96, 64, "f32"), (64, 96, "bf16"), (128, 128, "f32"), (768, 3072, "bf16"), (3072, 768, "bf16"),
          (96, 64, "bf16")]


def bound(precision, iters, k):
    e = {"fp32": 4.0 * math.sqrt(k) * 2.0 ** -24, "tf32": 4.0 * 2.0 ** -11, "bf16": 4.0 * 2.0 ** -8}[precision]
    return max(1e-6, 1.5 ** iters * e)


@pytest.mark.parametrize("precision", ["fp32", "tf32", "bf16"])
def test_muon_two_steps_against_oracle(dev, precision):
    import torch
    g = np.random.Generator(np.random.PCG64(17))
    iters = 5
    mats, host = [], []
    for m, n, gdt in SHAPES:
        X = g.normal(0, 0.02, (m, n)).astype(np.float32)
        grads = []
        for _ in range(2):
            Gn = (0.1 * g.standard_normal((m, n)) + g.standard_normal((m, 3)) @ g.standard_normal((3, n)) / 3)
            Gn = Gn.astype(np.float32)
            grads.append(synth.f32_to_bf16_bits(Gn) if gdt == "bf16" else Gn)
        Xd = torch.from_numpy(X).to(dev)
        mats.append(dict(X=Xd, G=grad_to_device(grads[0], dev), B=torch.zeros((m, n), device=dev),
                         eta=0.02, mu=0.95))
        host.append(dict(X=X.astype(np.float64), B=np.zeros((m, n)), grads=grads))
    plan = dion.MuonPlan(mats, iters=iters, precision=precision)
    assert plan.launches_per_step == 4 + iters * 3 * len({(m, n) for m, n, _ in SHAPES})
    worst = {}
    for t in range(2):
        for d, h in zip(mats, host):
            d["G"].copy_(grad_to_device(h["grads"][t], dev))
        X_before = [f64(d["X"]) for d in mats]
        B_before = [f64(d["B"]) for d in mats]
        plan.step()
        torch.cuda.synchronize()
        for k, (d, h) in enumerate(zip(mats, host)):
            m, n = d["X"].shape
            ref = MU.muon_step(X_before[k], f64(d["G"]), B_before[k], 0.02, 0.95, iters)
            dX = f64(d["X"]) - X_before[k]
            e = {"dX": rel(dX, ref["X"] - X_before[k]), "B": rel(f64(d["B"]), ref["B"])}
            tol = bound(precision, iters, max(m, n))
            assert e["B"] <= 1e-6 and e["dX"] <= tol, (m, n, precision, e, tol)
            for key, v in e.items():
                worst[key] = max(worst.get(key, 0.0), v)
    print(precision, "worst", worst)
    plan.close()
