"""The bounded-wait path of the tensor-core kernels (DION_MAT_TIMEOUT).

Every pipeline wait gives up after a time limit, raises the CTA's abort flag,
drains its own copies, frees TMEM and returns.  Through the testing hook
dion_debug_expire_wait the test lowers the limit to 100 ms and makes the
update kernel's operand producer withhold the operands of matrix 0, so that
the MMA issuer's wait on them runs out.  No fault and no endless wait is
involved: the wait ends by its limit.  Checked: matrix 0 reports
DION_MAT_TIMEOUT and its X and R are untouched (its only tile never ran); the
other matrices, whose tiles ran on other CTAs, are updated exactly as the
oracle says; and a normal step afterwards works.
"""
import numpy as np
import pytest

from parity_util import check_step, f64, state_snapshot
from rank_orthonormalized_optimizer_03_b300 import build, dion

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    dion.lib()
    return torch.device("cuda:0")


def make(dev, seed):
    import torch
    g = np.random.Generator(np.random.PCG64(seed))
    mats = []
    # one 128 x 128 update tile for matrix 0, two each for the others: five tiles,
    # one per CTA, so matrix 0's tile has a CTA of its own
    for m, n, r in [(128, 128, 16), (256, 128, 16), (128, 256, 32)]:
        mats.append(dict(X=torch.from_numpy(g.normal(0, 0.02, (m, n)).astype(np.float32)).to(dev),
                         G=torch.from_numpy(g.standard_normal((m, n)).astype(np.float32)).to(dev),
                         R=torch.zeros((m, n), device=dev),
                         V=torch.from_numpy(np.linalg.qr(g.standard_normal((n, r)))[0].astype(np.float32)).to(dev),
                         eta=0.02, beta=0.95, variant="orth"))
    return mats


def test_expired_wait_marks_timeout_and_the_gpu_stays_usable(dev):
    import torch
    mats = make(dev, 3)
    plan = dion.Plan(mats)
    before = [state_snapshot(d) for d in mats]
    x0, r0 = mats[0]["X"].clone(), mats[0]["R"].clone()
    dion.debug_expire_wait(100_000_000, 0)
    try:
        plan.step()
        torch.cuda.synchronize()
    finally:
        dion.debug_expire_wait()
        torch.cuda.synchronize()
    st = plan.status()
    assert st[0] & dion.DION_MAT_TIMEOUT, st
    assert st[1] == 0 and st[2] == 0, st
    assert torch.equal(mats[0]["X"], x0) and torch.equal(mats[0]["R"], r0)
    for k in (1, 2):
        check_step(before[k], f64(mats[k]["G"]), mats[k], 0.02, 0.95, "orth", U_gpu=plan.buffer(k, dion.BUF_U))
    plan.close()
    # the context is still usable: a normal step of fresh state matches the oracle
    fresh = make(dev, 4)
    p2 = dion.Plan(fresh)
    b2 = [state_snapshot(d) for d in fresh]
    p2.step()
    torch.cuda.synchronize()
    assert p2.status() == [0, 0, 0]
    for k in range(3):
        check_step(b2[k], f64(fresh[k]["G"]), fresh[k], 0.02, 0.95, "orth", U_gpu=p2.buffer(k, dion.BUF_U))
    p2.close()
