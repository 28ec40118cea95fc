"""The byte and flop accounting behind the bench's GB/s and roofline figures,
pinned to counts derived by hand from the shapes (CPU only)."""
import pytest

from rank_orthonormalized_optimizer_03_b300 import accounting, workloads


@pytest.mark.parametrize("g_dtype, gb, minimum, schedule", [("bf16", 2, 30, 30), ("f32", 4, 32, 36)])
def test_bytes_per_element_and_factor_traffic(g_dtype, gb, minimum, schedule):
    m, n, r = 3072, 8192, 192
    c = accounting.phase_cost(m, n, r, g_dtype, "orth")
    # this library's schedule: (G + R) read in (a) and (c), then G, R, X read and X, R written
    total = sum(v.bytes for v in c.values())
    assert total == m * n * schedule + 4 * r * (2 * m + 3 * n)
    assert c["a"].bytes == m * n * (gb + 4) + 4 * r * (n + m)
    assert c["e"].bytes == m * n * (gb + 4 + 4 + 8)
    # the algorithmic minimum: storing M (gb + 4 + 4, then 4, then 4 + 4 + 4 + 4) or re-forming it
    assert accounting.state_bytes_per_elem(g_dtype) == minimum
    assert accounting.step_algorithmic(m, n, r, g_dtype, "orth").bytes == m * n * minimum + 4 * r * (2 * m + 3 * n)


def test_flops_of_the_four_contractions_and_orth():
    m, n, r = 1000, 600, 40
    qr = lambda k: 2 * k * r * r - 2 * r ** 3 / 3
    orth = accounting.phase_cost(m, n, r, "bf16", "orth")
    dion = accounting.phase_cost(m, n, r, "bf16", "dion")
    assert orth["a"].flops + orth["c"].flops + orth["e"].flops == 8 * m * n * r
    assert orth["b"].flops == qr(m) and orth["d"].flops == qr(n)
    assert dion["d"].flops == 2 * n * r
    assert {k: v.bytes for k, v in orth.items()} == {k: v.bytes for k, v in dion.items()}


def test_workload_sizes_match_the_model_shapes():
    # 28 layers of q, o (3072^2), k, v (1024 x 3072), gate, up (8192 x 3072), down (3072 x 8192)
    per_layer = 2 * 3072 * 3072 + 2 * 1024 * 3072 + 2 * 8192 * 3072 + 3072 * 8192
    wl = workloads.llama_3b(16)
    assert len(wl.mats) == 196 and wl.elems == 28 * per_layer == 2_818_572_288
    assert sorted({s.r for s in wl.mats}) == [64, 192]
    assert sorted({s.r for s in workloads.llama_3b(4).mats}) == [256, 768]
    # 12 layers of 4 x 768^2, 3072 x 768, 768 x 3072
    g = workloads.gpt_160m(4)
    assert len(g.mats) == 72 and g.elems == 12 * (4 * 768 * 768 + 2 * 3072 * 768) == 84_934_656


def test_step_cost_of_the_benchmark_workload():
    wl = workloads.llama_3b(16)
    cost = accounting.step_cost(wl.mats, wl.g_dtype, lambda i: "orth")
    factors = sum(4 * s.r * (2 * s.m + 3 * s.n) for s in wl.mats)
    assert cost["step"].bytes == 30 * wl.elems + factors
    # 30 B per element and the factors: the 87.1 GB of the workload's byte budget
    assert abs(cost["step"].bytes / 1e9 - 87.1) < 0.1
    assert cost["a"].flops + cost["c"].flops + cost["e"].flops == sum(8 * s.m * s.n * s.r for s in wl.mats)
    impl = sum(30 * s.m * s.n + 4 * s.r * (5 * s.m + 6 * s.n) for s in wl.mats)
    assert cost["impl_extra_bytes"] == impl - cost["step"].bytes
