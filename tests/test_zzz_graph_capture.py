"""The step captured once into a CUDA graph and replayed (GPU).

`dion_step_batched` enqueues only kernel launches and one memset on the caller's
stream, and its kernels read the per-matrix tables (pointers, tensor maps, eta,
beta) from the workspace when they run.  So once `dion_plan_upload` has put the
tables in place outside the capture, every replay of a captured step is one
optimizer step.  A later `set_hparams` followed by an upload changes what the
replays do, without a new capture.  The replays are compared bit for bit with
eager steps on a copy of the same state.
"""
import numpy as np
import pytest

from parity_util import f64, orth_v0
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


def layer0_batch(dev):
    """The six matrices of GPT-160M's first layer, Orth-Dion and Dion alternating."""
    import torch
    wl = workloads.gpt_160m(4)
    mats = []
    for k, spec in enumerate(wl.mats[:6]):
        X0, V0_raw, G = synth.device_matrix_inputs(spec, wl, k, seed=0, device=dev)
        V0 = torch.from_numpy(np.ascontiguousarray(orth_v0(f64(V0_raw)), dtype=np.float32)).to(dev)
        mats.append(dict(X=X0, G=G, R=torch.zeros_like(X0), V=V0, eta=spec.eta, beta=spec.beta,
                         variant=("orth", "dion")[k % 2], scale=spec.scale))
    return mats


def copy_of(mats):
    return [{k: (v.clone() if hasattr(v, "clone") else v) for k, v in d.items()} for d in mats]


def assert_same_state(a, b):
    import torch
    for i, (da, db) in enumerate(zip(a, b)):
        for k in ("X", "R", "V"):
            assert torch.equal(da[k], db[k]), (i, k)


def test_graph_replays_equal_eager_steps(dev):
    import torch
    a = layer0_batch(dev)
    b = copy_of(a)
    pa, pb = dion.Plan(a), dion.Plan(b)
    pb.upload()
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pb.step()
    torch.cuda.synchronize()
    assert_same_state(a, b)            # the capture records the step without running it

    for _ in range(2):
        pa.step()
        graph.replay()
    torch.cuda.synchronize()
    assert pa.failures() == [0] * len(a)
    assert pb.failures() == [0] * len(b)
    assert_same_state(a, b)

    # new hyper-parameters reach the replays through an upload of the tables
    for i in range(len(a)):
        pa.set_hparams(i, 0.05, 0.5)
        pb.set_hparams(i, 0.05, 0.5)
    pb.upload()
    pa.step()
    graph.replay()
    torch.cuda.synchronize()
    assert pb.failures() == [0] * len(b)
    assert_same_state(a, b)
