"""Host-side checks of the C ABI (no GPU needed: nothing here launches work).

plan creation, validation, workspace layout and status strings are host
logic; the descriptors carry fake (never dereferenced) device addresses.
"""
import ctypes

import numpy as np

import pytest

from rank_orthonormalized_optimizer_03_b300 import build, dion


@pytest.fixture(scope="module")
def L():
    build.build()
    return dion.lib()


def test_library_exports_every_declared_symbol(L):
    names = dion.header_functions()
    assert len(names) >= 13
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", dion.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)
    assert L.dion_abi_version() == 1


BASE = 0x7F0000000000
SLOT = 1 << 32   # every buffer gets its own 4 GiB slot of fake address space


def fake_desc(k, m=64, n=32, r=8, **kw):
    d = dict(X=BASE + (4 * k) * SLOT, G=BASE + (4 * k + 1) * SLOT, R=BASE + (4 * k + 2) * SLOT,
             V=BASE + (4 * k + 3) * SLOT, m=m, n=n, r=r, ld_x=n, ld_g=n, ld_r=n, g_dtype=dion.DTYPE_BF16,
             variant=1, eta=0.01, beta=0.95, scale=0.0, reserved=0.0)
    d.update(kw)
    return dion.MatrixDesc(**d)


def create(L, descs):
    arr = (dion.MatrixDesc * len(descs))(*descs)
    ws = ctypes.c_size_t(0)
    plan = ctypes.c_void_p()
    code = L.dion_plan_create(arr, len(descs), ctypes.byref(ws), ctypes.byref(plan))
    return code, ws.value, plan


def test_valid_plan_and_layout(L):
    descs = [fake_desc(0), fake_desc(1, m=100, n=40, r=40), fake_desc(2, variant=0, r=1)]
    code, ws, plan = create(L, descs)
    assert code == dion.DION_OK, L.dion_last_error()
    assert ws > 0 and L.dion_plan_count(plan) == 3
    assert L.dion_plan_launches_per_step(plan) >= 10
    off, rows, cols, ld = ctypes.c_size_t(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    seen = []
    for i, d in enumerate(descs):
        for which, nrow in ((dion.BUF_P, d.m), (dion.BUF_U, d.m), (dion.BUF_W, d.n)):
            assert L.dion_plan_buffer(plan, i, which, ctypes.byref(off), ctypes.byref(rows),
                                      ctypes.byref(cols), ctypes.byref(ld)) == 0
            assert rows.value == nrow and cols.value == d.r and ld.value >= d.r and ld.value % 16 == 0
            assert off.value % 256 == 0 and off.value + rows.value * ld.value * 4 <= ws
            seen.append((off.value, off.value + rows.value * ld.value * 4))
    seen.sort()
    for a, b in zip(seen, seen[1:]):
        assert a[1] <= b[0], "workspace buffers overlap"
    assert L.dion_plan_buffer(plan, 3, 0, ctypes.byref(off), ctypes.byref(rows), ctypes.byref(cols),
                              ctypes.byref(ld)) == dion.DION_ERR_INVALID_ARG
    assert L.dion_plan_set_hparams(plan, 1, 0.5, 0.5) == 0
    assert L.dion_plan_set_hparams(plan, 7, 0.5, 0.5) == dion.DION_ERR_INVALID_ARG
    assert L.dion_plan_set_hparams(plan, 0, float("nan"), 0.5) == dion.DION_ERR_INVALID_ARG
    L.dion_plan_destroy(plan)


@pytest.mark.parametrize("bad, code", [
    (dict(r=0), dion.DION_ERR_INVALID_ARG),
    (dict(r=33), dion.DION_ERR_INVALID_ARG),            # r > min(m, n)
    (dict(m=0), dion.DION_ERR_INVALID_ARG),
    (dict(m=1 << 31), dion.DION_ERR_INVALID_ARG),      # rows index as int32 on the device
    (dict(ld_x=16), dion.DION_ERR_INVALID_ARG),         # ld < n
    (dict(g_dtype=7), dion.DION_ERR_INVALID_ARG),
    (dict(variant=3), dion.DION_ERR_INVALID_ARG),
    (dict(eta=float("inf")), dion.DION_ERR_INVALID_ARG),
    (dict(reserved=1.0), dion.DION_ERR_INVALID_ARG),
    (dict(X=0), dion.DION_ERR_INVALID_ARG),
    (dict(X=BASE + 4), dion.DION_ERR_UNSUPPORTED),       # misaligned pointer
    (dict(ld_x=33), dion.DION_ERR_UNSUPPORTED),          # row pitch not 16-byte multiple
    (dict(ld_g=36), dion.DION_ERR_UNSUPPORTED),          # bf16 pitch 72 bytes
])
def test_invalid_descriptors_rejected(L, bad, code):
    got, _, plan = create(L, [fake_desc(0, **bad)])
    assert got == code, (bad, L.dion_last_error())
    assert not plan.value
    assert L.dion_last_error().decode() != ""


def test_overlapping_buffers_rejected(L):
    a = fake_desc(0)
    b = fake_desc(1, X=a.R + 128)          # X of matrix 1 inside R of matrix 0
    assert create(L, [a, b])[0] == dion.DION_ERR_INVALID_ARG
    c = fake_desc(1, G=a.G)                 # two matrices may share a read-only gradient
    assert create(L, [a, c])[0] == dion.DION_OK
    d = fake_desc(1, G=a.V)                 # but a gradient may not alias writable state
    assert create(L, [a, d])[0] == dion.DION_ERR_INVALID_ARG


def test_null_and_count_arguments(L):
    ws = ctypes.c_size_t(0)
    plan = ctypes.c_void_p()
    arr = (dion.MatrixDesc * 1)(fake_desc(0))
    assert L.dion_plan_create(None, 1, ctypes.byref(ws), ctypes.byref(plan)) == dion.DION_ERR_INVALID_ARG
    assert L.dion_plan_create(arr, 0, ctypes.byref(ws), ctypes.byref(plan)) == dion.DION_ERR_INVALID_ARG
    assert L.dion_plan_count(None) == -1
    L.dion_plan_destroy(None)


def test_launching_calls_check_workspace_before_touching_cuda(L):
    code, ws, plan = create(L, [fake_desc(0)])
    assert code == 0
    assert L.dion_step_batched(plan, None, ws, None) == dion.DION_ERR_WORKSPACE
    assert L.dion_step_batched(plan, 0x10000, ws - 1, None) == dion.DION_ERR_WORKSPACE
    assert L.dion_step_batched(plan, 0x10010, ws, None) == dion.DION_ERR_WORKSPACE   # misaligned
    assert L.dion_step_phases(plan, 0x10000, ws, 3, 1, None) == dion.DION_ERR_INVALID_ARG
    L.dion_plan_destroy(plan)


def test_status_strings(L):
    for code, name in dion.STATUS_NAMES.items():
        assert L.dion_status_string(code).decode() == name
    assert L.dion_status_string(99).decode() == "DION_ERR_UNKNOWN"


def plan_of(L, shapes):
    """Create (and destroy) a plan over fake buffers: (m, n, r, variant, g_dtype)."""
    descs = [fake_desc(k, m=m, n=n, r=r, ld_x=n, ld_g=n, ld_r=n, variant=v, g_dtype=gd)
             for k, (m, n, r, v, gd) in enumerate(shapes)]
    code, ws, plan = create(L, descs)
    msg = L.dion_last_error()
    if code == dion.DION_OK:
        L.dion_plan_destroy(plan)
    return code, ws, msg


@pytest.mark.parametrize("name", ["single_256x128_r16", "square_1024_r256", "gpt160m_12L_rdiv4",
                                  "llama3b_28L_rdiv16", "llama3b_28L_rdiv4", "sweep_8192x8192_r2048",
                                  "sweep_4096x16384_r32", "sweep_4096x16384_r1024"])
def test_work_tables_pass_their_check_for_every_workload(L, name):
    # dion_plan_create checks its work tables (coverage of every launch, K
    # ranges, 16-byte TMA x coordinates) before returning DION_OK
    from rank_orthonormalized_optimizer_03_b300 import workloads
    wl = workloads.by_name(name)
    bf = dion.DTYPE_BF16 if wl.g_dtype == "bf16" else dion.DTYPE_F32
    code, ws, msg = plan_of(L, [(s.m, s.n, s.r, k % 2, bf) for k, s in enumerate(wl.mats)])
    assert code == dion.DION_OK, msg
    assert ws > 0


def test_work_tables_pass_their_check_for_odd_batches(L):
    g = np.random.Generator(np.random.PCG64(5))
    for trial in range(40):
        shapes = []
        for _ in range(int(g.integers(1, 6))):
            m = int(g.integers(1, 700))
            n = int(g.integers(1, 90)) * 8          # bf16 / fp32 row pitches on 16 bytes
            r = int(g.integers(1, min(m, n) + 1))
            shapes.append((m, n, r, int(g.integers(0, 2)), int(g.integers(0, 2))))
        code, _, msg = plan_of(L, shapes)
        assert code == dion.DION_OK, (shapes, msg)


def muon_desc(k, m=64, n=32, **kw):
    d = dict(X=BASE + (3 * k) * SLOT, G=BASE + (3 * k + 1) * SLOT, B=BASE + (3 * k + 2) * SLOT, m=m, n=n,
             ld_x=n, ld_g=n, ld_b=n, g_dtype=dion.DTYPE_BF16, eta=0.01, mu=0.95, scale=0.0)
    d.update(kw)
    return dion.MuonDesc(**d)


def muon_create(L, descs, iters=5, precision=0, row_fraction=1.0):
    arr = (dion.MuonDesc * len(descs))(*descs)
    ws = ctypes.c_size_t(0)
    plan = ctypes.c_void_p()
    code = L.muon_plan_create(arr, len(descs), iters, precision, row_fraction, ctypes.byref(ws), ctypes.byref(plan))
    return code, ws.value, plan


def test_muon_plan_groups_shapes_and_validates(L):
    descs = [muon_desc(0), muon_desc(1), muon_desc(2, m=32, n=64), muon_desc(3, g_dtype=dion.DTYPE_F32)]
    code, ws, plan = muon_create(L, descs, iters=5)
    assert code == dion.DION_OK, L.dion_last_error()
    # two groups of equal shape (64 x 32: matrices 0, 1, 3; 32 x 64: matrix 2):
    # 4 streaming launches + 5 iterations x (2 GEMMs + diagonal) x 2 groups
    assert L.muon_plan_launches_per_step(plan) == 4 + 5 * 3 * 2
    # two ping-pong Y buffers (bf16) of 4 matrices of 2048 elements, the Grams, 32 MB of GEMM scratch
    assert ws >= (32 << 20) + 2 * 2 * 4 * 2048
    L.muon_plan_destroy(plan)
    for bad, kw in [("precision", dict(precision=3)), ("iters", dict(iters=-1))]:
        code, _, _ = muon_create(L, descs, **kw)
        assert code == dion.DION_ERR_INVALID_ARG, bad
    for kw in [dict(X=0), dict(ld_b=16), dict(g_dtype=7), dict(m=0)]:
        code, _, _ = muon_create(L, [muon_desc(0, **kw)])
        assert code == dion.DION_ERR_INVALID_ARG, kw
    L.muon_plan_destroy(None)


def test_row_selection_plan(L):
    descs = [muon_desc(0, m=100, n=32), muon_desc(1, m=64, n=32)]
    code, ws, plan = muon_create(L, descs, iters=3, row_fraction=0.25)
    assert code == dion.DION_OK, L.dion_last_error()
    # k = ceil(0.25 m): 25 and 16 rows -> two groups (25 x 32, 16 x 32)
    assert L.muon_plan_launches_per_step(plan) == 5 + 3 * 3 * 2
    off, k = ctypes.c_size_t(), ctypes.c_int64()
    assert L.muon_plan_selected_rows(plan, 0, ctypes.byref(off), ctypes.byref(k)) == dion.DION_OK and k.value == 25
    assert L.muon_plan_selected_rows(plan, 1, ctypes.byref(off), ctypes.byref(k)) == dion.DION_OK and k.value == 16
    assert L.muon_plan_selected_rows(plan, 2, ctypes.byref(off), ctypes.byref(k)) == dion.DION_ERR_INVALID_ARG
    L.muon_plan_destroy(plan)
    for rf in (0.0, 1.5, float("nan")):
        assert muon_create(L, descs, row_fraction=rf)[0] == dion.DION_ERR_INVALID_ARG, rf
    assert muon_create(L, [muon_desc(0, m=20000, n=32)], row_fraction=0.5)[0] == dion.DION_ERR_UNSUPPORTED
    code, _, plan = muon_create(L, descs)
    assert L.muon_plan_selected_rows(plan, 0, ctypes.byref(off), ctypes.byref(k)) == dion.DION_ERR_INVALID_ARG
    L.muon_plan_destroy(plan)


@pytest.mark.parametrize("shapes", [[(8192, 8192, 2048)], [(3072, 3072, 768), (1024, 3072, 256), (8192, 3072, 768)],
                                    [(1200, 640, 300), (200, 160, 16)]])
def test_large_rank_plans_pass_their_table_checks(L, shapes):
    """Ranks above 192 take the blocked-Cholesky orth() path: its Gram items (transposed
    streaming mode, K split over rows) pass the plan's coverage checks."""
    descs = [fake_desc(k, m=m, n=n, r=r, variant=k % 2) for k, (m, n, r) in enumerate(shapes)]
    code, ws, plan = create(L, descs)
    assert code == dion.DION_OK, L.dion_last_error()
    rmax = max(r for _, _, r in shapes)
    np_ = -(-rmax // 128)
    # at least three CholeskyQR passes of (Gram, reduce, np panels, inverse, split, A T) for orth(P)
    assert L.dion_plan_launches_per_step(plan) > 3 * (4 + np_)
    L.dion_plan_destroy(plan)


@pytest.mark.parametrize("name, launches", [("llama3b_28L_rdiv16", 28), ("gpt160m_12L_rdiv4", 29)])
def test_model_batch_launches_and_w_split(L, name, launches):
    """Launches of one Orth-Dion step of the model batches: (a) split + stream, orth(P)
    in three CholeskyQR passes of four launches, (c) stream (+ the reduction of W's
    K-range partials only where phase (c) splits K), orth(W), one update launch.  The
    Llama-3B batch has items enough to fill the GPU and none above its row cap; the
    GPT-160M batch splits the K of its 3072-row matrices, which exceed the cap of
    2048 rows (a third of a CTA's share of its work is less than that)."""
    from rank_orthonormalized_optimizer_03_b300 import workloads
    wl = workloads.by_name(name)
    descs = [fake_desc(k, m=s.m, n=s.n, r=s.r, variant=1) for k, s in enumerate(wl.mats)]
    code, ws, plan = create(L, descs)
    assert code == dion.DION_OK, L.dion_last_error()
    assert L.dion_plan_launches_per_step(plan) == launches
    L.dion_plan_destroy(plan)


def test_work_tables_pass_their_check_for_odd_large_rank_batches(L):
    # ranks above 192 take the blocked orth() (tiled Gram, Cholesky across the GPU,
    # inverse by recursive doubling) and ranks above 256 several update launches;
    # ragged m, n and r exercise the tail tiles of every one of their tables; one
    # large rank puts the whole batch, small ranks included, on the blocked orth()
    g = np.random.Generator(np.random.PCG64(11))
    for trial in range(24):
        shapes = []
        for j in range(int(g.integers(1, 5))):
            m = int(g.integers(193, 9000))
            n = int(g.integers(25, 1100)) * 8
            r = int(g.integers(193 if j == 0 else 1, min(m, n, 2048) + 1))
            shapes.append((m, n, r, int(g.integers(0, 2)), int(g.integers(0, 2))))
        code, ws, msg = plan_of(L, shapes)
        assert code == dion.DION_OK, (shapes, msg)
        assert ws > 0


def test_last_error_is_per_host_thread(L):
    """dion_last_error() keeps each host thread's own message: two threads fail plan
    creation for different reasons at once and each reads back its own reason."""
    import threading
    barrier = threading.Barrier(2)
    seen = {}

    def worker(name, desc):
        arr = (dion.MatrixDesc * 1)(desc)
        ws, plan = ctypes.c_size_t(0), ctypes.c_void_p()
        for _ in range(200):
            barrier.wait()
            code = L.dion_plan_create(arr, 1, ctypes.byref(ws), ctypes.byref(plan))
            barrier.wait()
            msg = L.dion_last_error().decode()
            seen.setdefault(name, set()).add((code, msg))

    t1 = threading.Thread(target=worker, args=("rank", fake_desc(0, r=40)))
    t2 = threading.Thread(target=worker, args=("dtype", fake_desc(0, g_dtype=9)))
    t1.start(); t2.start(); t1.join(); t2.join()
    assert len(seen["rank"]) == 1 and len(seen["dtype"]) == 1, seen
    (c1, m1), = seen["rank"]
    (c2, m2), = seen["dtype"]
    assert c1 == c2 == dion.DION_ERR_INVALID_ARG
    assert "rank" in m1 and "dtype" in m2, (m1, m2)


def test_exchange_regions_of_the_sharded_step(L):
    """dion_plan_exchange: the W region is every matrix's n x rp W back to back in plan
    order (the buffers dion_plan_buffer reports), the Gram region every rp x rp Gram;
    both aligned, inside the workspace and apart from each other and from P and U."""
    shapes = [(100, 40, 40), (64, 96, 7), (300, 128, 33), (17, 24, 1)]
    descs = [fake_desc(k, m=m, n=n, r=r) for k, (m, n, r) in enumerate(shapes)]
    code, ws, plan = create(L, descs)
    assert code == dion.DION_OK, L.dion_last_error()
    rp = [-(-r // 32) * 32 for _, _, r in shapes]
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.dion_plan_exchange(plan, 1, ctypes.byref(off), ctypes.byref(nb)) == dion.DION_OK
    w_off, w_bytes = off.value, nb.value
    assert w_bytes == sum(4 * n * q for (_, n, _), q in zip(shapes, rp))
    assert L.dion_plan_exchange(plan, 0, ctypes.byref(off), ctypes.byref(nb)) == dion.DION_OK
    g_off, g_bytes = off.value, nb.value
    assert g_bytes == sum(4 * q * q for q in rp)
    for o, b in ((w_off, w_bytes), (g_off, g_bytes)):
        assert o % 16 == 0 and o + b <= ws
    assert w_off + w_bytes <= g_off or g_off + g_bytes <= w_off
    bo, rows, cols, ld = ctypes.c_size_t(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    expect = w_off
    for i, (m, n, r) in enumerate(shapes):
        assert L.dion_plan_buffer(plan, i, dion.BUF_W, ctypes.byref(bo), ctypes.byref(rows), ctypes.byref(cols),
                                  ctypes.byref(ld)) == dion.DION_OK
        assert (bo.value, rows.value, cols.value, ld.value) == (expect, n, r, rp[i])
        expect += 4 * n * rp[i]
        for which in (dion.BUF_P, dion.BUF_U):
            assert L.dion_plan_buffer(plan, i, which, ctypes.byref(bo), ctypes.byref(rows), ctypes.byref(cols),
                                      ctypes.byref(ld)) == dion.DION_OK
            lo, hi = bo.value, bo.value + 4 * m * rp[i]
            for o, b in ((w_off, w_bytes), (g_off, g_bytes)):
                assert hi <= o or o + b <= lo
    assert L.dion_plan_exchange(plan, 2, ctypes.byref(off), ctypes.byref(nb)) == dion.DION_ERR_INVALID_ARG
    assert L.dion_plan_exchange(plan, 0, None, ctypes.byref(nb)) == dion.DION_ERR_INVALID_ARG
    L.dion_plan_destroy(plan)
