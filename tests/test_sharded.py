"""Row-sharded Dion / Orth-Dion step (rank_orthonormalized_optimizer_03_b300.sharded).

CPU: the orchestration ``sharded_step`` with the float64 shard backend, on
ranks emulated in one process and on two real gloo ranks, against the
unsharded float64 oracle step of the whole matrix; a dropped exchange is
caught.  GPU: the library's staged step (dion_shard_stage) with 1, 2 and 3
row shards emulated on one device against the oracle, and one rank's staged
step against the fused dion_step_batched (bitwise on the tensor-core path).
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from oracle import dion_oracle as O
from oracle.dion_sharded import ShardBackend
from parity_util import TOL_DX, TOL_STEP, f64, factor_tolerance, grad_to_device, rel
from rank_orthonormalized_optimizer_03_b300 import build, dion, synth
from rank_orthonormalized_optimizer_03_b300.sharded import (EmulatedRanks, ShardPlan, row_bounds, sharded_step,
                                                            EXCHANGE_AFTER)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def problem(m, n, r, seed):
    """A gradient of rank-3 signal plus noise of comparable size, so that the
    residual beyond rank r is not a tiny difference of large terms (its relative
    error would then measure fp32 rounding of M, not the sharding)."""
    g = np.random.Generator(np.random.PCG64(seed))
    X = g.normal(0, 0.02, (m, n))
    R = 0.05 * g.standard_normal((m, n))
    G = g.standard_normal((m, 3)) @ g.standard_normal((3, n)) + 0.5 * g.standard_normal((m, n))
    V = g.standard_normal((n, r)) / math.sqrt(n)
    return X, G, R, V


def local_allreduce(backends):
    """In-process stand-in for an all-reduce over the given backends."""
    def run():
        for k in range(5):
            for b in backends:
                b.stage(k)
            if k in EXCHANGE_AFTER:
                bufs = [b.exchange(EXCHANGE_AFTER[k]) for b in backends]
                tot = sum(x.clone() for x in bufs)
                for x in bufs:
                    x.copy_(tot)
    return run


@pytest.mark.parametrize("ranks", [1, 2, 3])
@pytest.mark.parametrize("variant", [O.ORTH, O.DION])
def test_float64_shards_equal_the_unsharded_step(ranks, variant):
    m, n, r = 90, 40, 6
    X, G, R, V = problem(m, n, r, seed=ranks)
    s = math.sqrt(m / n)
    ref = O.oracle_step(X, G, R, V, 0.03, 0.9, variant, s)
    bks = [ShardBackend(X[a:b], G[a:b], R[a:b], V, 0.03, 0.9, variant, s) for a, b in row_bounds(m, ranks)]
    local_allreduce(bks)()
    assert np.abs(np.vstack([b.X for b in bks]) - ref["X"]).max() < 1e-12
    assert np.abs(np.vstack([b.R for b in bks]) - ref["R"]).max() < 1e-12
    for b in bks:
        assert np.abs(b.V - ref["V"]).max() < 1e-11


def test_dropped_exchange_is_caught():
    """Skipping the all-reduce of W (or of the Grams) gives a different step."""
    m, n, r = 90, 40, 6
    X, G, R, V = problem(m, n, r, seed=5)
    ref = O.oracle_step(X, G, R, V, 0.03, 0.9, O.ORTH, 1.0)
    for skip in ("gram", "w"):
        bks = [ShardBackend(X[a:b], G[a:b], R[a:b], V, 0.03, 0.9, O.ORTH, 1.0) for a, b in row_bounds(m, 2)]
        for k in range(5):
            for b in bks:
                b.stage(k)
            if k in EXCHANGE_AFTER and EXCHANGE_AFTER[k] != skip:
                bufs = [b.exchange(EXCHANGE_AFTER[k]) for b in bks]
                tot = sum(x.clone() for x in bufs)
                for x in bufs:
                    x.copy_(tot)
        assert np.abs(np.vstack([b.X for b in bks]) - ref["X"]).max() > 1e-6, skip


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _gloo_rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from oracle.dion_sharded import ShardBackend as SB
    from rank_orthonormalized_optimizer_03_b300.sharded import dist_allreduce, row_bounds as rb, sharded_step as step
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m, n, r = 70, 30, 5
        X, G, R, V = problem(m, n, r, seed=9)
        a, b = rb(m, world)[rank]
        bk = SB(X[a:b], G[a:b], R[a:b], V, 0.02, 0.95, "orth", math.sqrt(m / n))
        for _ in range(2):                       # two chained steps: V and R carried
            step(bk, dist_allreduce())
        out[rank] = (bk.X, bk.R, bk.V)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_match_the_unsharded_chain():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_gloo_rank, args=(world, port, out), nprocs=world, join=True)
    m, n, r = 70, 30, 5
    X, G, R, V = problem(m, n, r, seed=9)
    steps = O.oracle_chain(X, R, V, [G, G], 0.02, 0.95, O.ORTH, math.sqrt(m / n))
    Xs = np.vstack([out[k][0] for k in range(world)])
    Rs = np.vstack([out[k][1] for k in range(world)])
    assert np.abs(Xs - steps[-1]["X"]).max() < 1e-12
    assert np.abs(Rs - steps[-1]["R"]).max() < 1e-12
    assert np.abs(out[0][2] - out[1][2]).max() == 0.0          # V replicated, identical on both ranks
    assert np.abs(out[0][2] - steps[-1]["V"]).max() < 1e-11


# ---------------------------------------------------------------- GPU
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


CASES = [(1000, 512, 32, "orth", "bf16"), (768, 600, 48, "dion", "f32"), (3072, 768, 192, "orth", "bf16"),
         (1200, 640, 300, "orth", "bf16")]


@pytest.mark.gpu
@pytest.mark.parametrize("ranks", [1, 2, 3])
@pytest.mark.parametrize("m,n,r,variant,gdt", CASES)
def test_emulated_gpu_ranks_against_oracle(dev, ranks, m, n, r, variant, gdt):
    import torch
    X, Gn, R, V = problem(m, n, r, seed=m + r)
    G = synth.f32_to_bf16_bits(Gn.astype(np.float32)) if gdt == "bf16" else Gn.astype(np.float32)
    X32, R32, V32 = (a.astype(np.float32) for a in (X, R, V))
    G64 = synth.bf16_bits_to_f32(G).astype(np.float64) if gdt == "bf16" else G.astype(np.float64)
    s = math.sqrt(m / n)
    ref = O.oracle_step(X32, G64, R32, V32, 0.02, 0.95, variant, s, qr=O.lapack_qr_pos)
    shards = []
    for a, b in row_bounds(m, ranks):
        shards.append(dict(X=to_dev(X32[a:b], dev), G=grad_to_device(np.ascontiguousarray(G[a:b]), dev),
                           R=to_dev(R32[a:b], dev), V=to_dev(V32, dev), eta=0.02, beta=0.95, variant=variant))
    plans = [ShardPlan([d], [m]) for d in shards]
    emu = EmulatedRanks(plans)
    emu.step()
    torch.cuda.synchronize()
    for st in emu.status():
        assert [v & dion.FATAL for v in st] == [0]
    Xg = np.vstack([f64(d["X"]) for d in shards])
    Rg = np.vstack([f64(d["R"]) for d in shards])
    errs = {"X": rel(Xg, ref["X"]), "R": rel(Rg, ref["R"]), "dX": rel(Xg - X32, ref["X"] - X32),
            "V": rel(f64(shards[0]["V"]), ref["V"]), "tol_V": factor_tolerance(ref)}
    assert errs["X"] <= TOL_STEP and errs["R"] <= TOL_STEP and errs["dX"] <= TOL_DX, errs
    assert errs["V"] <= errs["tol_V"], errs
    for d in shards[1:]:
        assert torch.equal(d["V"], shards[0]["V"])              # every rank holds the same Vbar
    print(m, n, r, variant, ranks, errs)
    for p in plans:
        p.close()


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["orth", "dion"])
def test_one_rank_staged_step_equals_fused_step(dev, variant):
    """On the tensor-core path (r <= 192) the stages run the fused step's kernels
    in the fused step's order, so one rank's staged step is bitwise the fused step."""
    import torch
    m, n, r = 1024, 768, 64
    X, Gn, R, V = problem(m, n, r, seed=77)
    a = dict(X=to_dev(X, dev), G=to_dev(Gn, dev), R=to_dev(R, dev), V=to_dev(V, dev), eta=0.02, beta=0.95,
             variant=variant, scale=math.sqrt(m / n))
    b = {k: (v.clone() if hasattr(v, "clone") else v) for k, v in a.items()}
    pa, pb = dion.Plan([a]), ShardPlan([b], [m])
    for _ in range(2):
        pa.step()
        sharded_step(pb, lambda t: None)             # one rank: the all-reduce is the identity
    torch.cuda.synchronize()
    for k in ("X", "R", "V"):
        assert torch.equal(a[k], b[k]), k
    pa.close()
    pb.close()
