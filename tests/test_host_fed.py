"""Host-fed steps (gradients copied from pinned host memory every step, in
groups whose copies overlap the previous group's step): the grouping on the
CPU, and on the GPU the same results as one plan over the whole batch."""
import math

import pytest

from parity_util import f64, rel
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth, workloads
from rank_orthonormalized_optimizer_03_b300.dion import group_bounds


@pytest.mark.parametrize("sizes, groups", [
    ([1] * 10, 3), ([5, 1, 1, 1, 1, 1], 3), ([1, 1], 5), ([3], 2), ([1] * 196, 14),
    ([2, 2, 8, 8, 8, 8, 2], 7), ([7, 1, 1, 1, 1, 1, 1, 1], 4)])
def test_group_bounds_cover_in_order_and_balance(sizes, groups):
    rg = group_bounds(sizes, groups)
    assert rg[0][0] == 0 and rg[-1][1] == len(sizes)
    assert all(a < b for a, b in rg)
    assert all(rg[k][1] == rg[k + 1][0] for k in range(len(rg) - 1))
    assert len(rg) <= min(groups, len(sizes))
    if groups <= len(sizes):
        # no range exceeds its share by more than its largest item
        share = sum(sizes) / len(rg)
        assert all(sum(sizes[a:b]) <= share + max(sizes) for a, b in rg)


@pytest.mark.gpu
def test_host_fed_groups_match_one_plan():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dev = torch.device("cuda:0")
    wl = workloads.gpt_160m(4)

    def state():
        mats = []
        for k, spec in enumerate(wl.mats):
            X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, k, seed=3, device=dev)
            mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=(V0_raw / math.sqrt(spec.n)).contiguous(),
                             eta=spec.eta, beta=spec.beta, variant=("orth", "dion")[k % 2], scale=spec.scale))
        return mats

    ref = state()
    fed = state()
    plan = dion.Plan(ref)
    # two groups of six layers each still fill the GPU, so every matrix gets
    # the same K split of W = M^T U as in the single plan
    stepper = dion.HostFedStep(fed, groups=2)
    assert len(stepper.plans) == 2 and len(stepper.host_slabs) == 2
    for i, d in enumerate(fed):
        stepper.host_grad(i).copy_(d["G"].cpu())
        assert stepper.host_grad(i).is_pinned()
    for slab in stepper.dev_slabs:
        slab.zero_()              # the host copy must bring the gradients in
    for _ in range(2):            # the second step waits for the first one's reads
        plan.step()
        stepper.step()
    torch.cuda.synchronize()
    assert plan.failures() == [0] * len(ref)
    assert [v & dion.FATAL for v in stepper.status()] == [0] * len(fed)
    for i, d in enumerate(ref):
        assert torch.equal(stepper.mats[i]["G"], d["G"])
    worst = 0.0
    for a, b in zip(ref, stepper.mats):
        for key in ("X", "R", "V"):
            worst = max(worst, rel(f64(b[key]), f64(a[key])))
    assert worst <= 1e-6, worst
    print("largest relative difference", worst)
    stepper.close()
    plan.close()
