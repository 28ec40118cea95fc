"""Algorithmic bytes and flops of the Dion / Orth-Dion step (host arithmetic only).

Bytes per element of an m x n matrix for the three streaming passes (M is
recomputed from G + R in every pass instead of being stored):

  (a) P = (G + R) V            reads G, R                     gb + 4
  (c) W = (G + R)^T U          reads G, R                     gb + 4
  (e) X -= eta s U Vbar^T,     reads G, R, X; writes X, R     gb + 4 + 4 + 8
      R  = beta (G + R - U W^T)
  total = 3 gb + 24  (30 B with a bf16 gradient, 36 B with fp32)

The alternative of storing M in pass (a) costs the same (gb + 4 + 4, then
4, then 4 + 4 + 8 = gb + 28 ... = 30 B for bf16 G) so either schedule's
minimum is 30 B/element for bf16 G.  The factors add 4 r (5 m + 6 n) bytes:
(a) reads V, writes P; orth(P) reads P, writes U; (c) reads U, writes W;
orth(W) / colnorm reads W, writes Vbar; (e) reads U, Vbar and W.

Flops per matrix: 8 m n r for the four contractions (M V, M^T U, U Vbar^T,
U W^T), plus 2 m r^2 - 2/3 r^3 for orth(P) (Householder count), plus
2 n r^2 - 2/3 r^3 for orth(W) (Orth-Dion) or 3 n r for the column norms
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


def phase_cost(m: int, n: int, r: int, g_dtype: str, variant: str) -> dict:
    gb = gbytes(g_dtype)
    e = m * n
    qr = lambda k: 2.0 * k * r * r - 2.0 * r ** 3 / 3.0
    return {
        "a": Cost(e * (gb + 4) + 4.0 * (n * r + m * r), 2.0 * e * r),
        "b": Cost(4.0 * 2 * m * r, qr(m)),
        "c": Cost(e * (gb + 4) + 4.0 * (m * r + n * r), 2.0 * e * r),
        "d": Cost(4.0 * 2 * n * r, qr(n) if variant == "orth" else 3.0 * n * r),
        "e": Cost(e * (gb + 16) + 4.0 * (m * r + 2 * n * r), 4.0 * e * r),
    }


def step_cost(mats: Iterable, g_dtype: str, variant_of) -> dict:
    tot = {k: Cost() for k in "abcde"}
    for i, s in enumerate(mats):
        pc = phase_cost(s.m, s.n, s.r, g_dtype, variant_of(i))
        for k in tot:
            tot[k] = tot[k] + pc[k]
    tot["step"] = sum((tot[k] for k in "abcde"), Cost())
    return tot
