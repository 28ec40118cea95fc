"""Algorithmic bytes and flops of the Dion / Orth-Dion step (host arithmetic only).

Two byte counts per element of an m x n matrix are kept apart.

The ALGORITHMIC count is the least traffic any schedule of the step needs:
M must be touched in three passes (P = M V, then W = M^T U, then the update),
because orth() sits between them.  Either M is stored by pass (a) and read back,
or it is re-formed from G + R in every pass:

  store M:      (a) G gb + R 4 + M 4,  (c) M 4,   (e) M 4 + X 4 + X 4 + R 4   = gb + 28
  recompute M:  (a) G gb + R 4,        (c) G gb + R 4,  (e) G gb + R 4 + X 8 + R 4 = 3 gb + 24

so the minimum is min(gb + 28, 3 gb + 24): 30 B with a bf16 gradient (both
schedules), 32 B with fp32 (storing M).  The factors add 4 r (2 m + 3 n) bytes
per matrix: V read and P written (a), U read and W written (c), Vbar written (d).
These are the bytes behind the step's GB/s and its roofline.

The SCHEDULE count is what each kernel of this library must move under its own
schedule (M re-formed in every pass): (a) and (c) gb + 4, (e) gb + 16 per
element (36 B in all with fp32 G), with the factor bytes of the minimum above
attributed to the phases that read or write them.  The per-kernel rooflines
use these.  ``impl_factor_bytes`` is the factor traffic the present kernels
make (P, U, W written once and read back, and the tf32 operand halves the
tensor cores read), reported apart as an implementation cost.

Flops per matrix: 8 m n r for the four contractions (M V, M^T U, U Vbar^T,
U W^T), plus 2 m r^2 - 2/3 r^3 for orth(P) (Householder count), plus
2 n r^2 - 2/3 r^3 for orth(W) (Orth-Dion) or 2 n r for the column norms
(Dion).  CholeskyQR2's extra Gram work is an implementation cost and is not
counted.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Iterable


@dataclass
class Cost:
    bytes: float = 0.0
    flops: float = 0.0

    def __add__(self, o):
        return Cost(self.bytes + o.bytes, self.flops + o.flops)


def gbytes(g_dtype: str) -> int:
    return 2 if g_dtype == "bf16" else 4


def state_bytes_per_elem(g_dtype: str) -> int:
    """The algorithmic minimum per element: min(store M, re-form M)."""
    gb = gbytes(g_dtype)
    return min(gb + 28, 3 * gb + 24)


def factor_bytes(m: int, n: int, r: int) -> float:
    """Least factor traffic: V, U read; P, W, Vbar written (each once)."""
    return 4.0 * r * (2 * m + 3 * n)


def impl_factor_bytes(m: int, n: int, r: int) -> float:
    """Factor traffic of the present kernels, without the tf32 halves: (a) reads V,
    writes P; orth(P) reads P, writes U; (c) reads U, writes W; orth(W) / colnorm
    reads W, writes Vbar; (e) reads U, Vbar and W."""
    return 4.0 * r * (5 * m + 6 * n)


def phase_cost(m: int, n: int, r: int, g_dtype: str, variant: str) -> dict:
    """Per-phase cost under this library's schedule (M re-formed in every pass)."""
    gb = gbytes(g_dtype)
    e = m * n
    qr = lambda k: 2.0 * k * r * r - 2.0 * r ** 3 / 3.0
    return {
        "a": Cost(e * (gb + 4) + 4.0 * (n * r + m * r), 2.0 * e * r),
        "b": Cost(0.0, qr(m)),
        "c": Cost(e * (gb + 4) + 4.0 * (m * r + n * r), 2.0 * e * r),
        "d": Cost(4.0 * n * r, qr(n) if variant == "orth" else 2.0 * n * r),
        "e": Cost(e * (gb + 16), 4.0 * e * r),
    }


def step_algorithmic(m: int, n: int, r: int, g_dtype: str, variant: str) -> Cost:
    """The step's algorithmic bytes (the minimum above) and flops for one matrix."""
    flops = sum(c.flops for c in phase_cost(m, n, r, g_dtype, variant).values())
    return Cost(m * n * state_bytes_per_elem(g_dtype) + factor_bytes(m, n, r), flops)


def step_cost(mats: Iterable, g_dtype: str, variant_of) -> dict:
    """Per-phase schedule costs, summed over the matrices, plus "step" (the
    algorithmic minimum of the whole step) and "impl_extra_bytes" (what the
    present kernels move beyond it, tf32 halves not included)."""
    tot = {k: Cost() for k in "abcde"}
    step = Cost()
    extra = 0.0
    for i, s in enumerate(mats):
        pc = phase_cost(s.m, s.n, s.r, g_dtype, variant_of(i))
        for k in tot:
            tot[k] = tot[k] + pc[k]
        step = step + step_algorithmic(s.m, s.n, s.r, g_dtype, variant_of(i))
        extra += (s.m * s.n * (3 * gbytes(g_dtype) + 24) + impl_factor_bytes(s.m, s.n, s.r)) \
            - (s.m * s.n * state_bytes_per_elem(g_dtype) + factor_bytes(s.m, s.n, s.r))
    tot["step"] = step
    tot["impl_extra_bytes"] = extra
    return tot
