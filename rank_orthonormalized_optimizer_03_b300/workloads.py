"""Workload definitions: matrix shapes, ranks and hyper-parameters.

Plain data, no arithmetic of the method.  Each workload is a list of
``MatrixSpec`` (one per weight matrix, in the order the step processes them)
plus the gradient recipe that ``synth`` uses to fill it.

Shapes follow PyTorch's ``(out_features, in_features)`` convention, so a
matrix is m x n with m = out, n = in.  The rank of each matrix is
``max(1, min(m, n) // rank_div)`` unless a workload fixes it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional


@dataclass(frozen=True)
class MatrixSpec:
    name: str
    m: int
    n: int
    r: int
    eta: float
    beta: float
    scale: float          # s in X <- X - eta*s*U Vbar^T; sqrt(m/n) by default

    @property
    def elems(self) -> int:
        return self.m * self.n


@dataclass(frozen=True)
class Workload:
    name: str
    mats: List[MatrixSpec]
    g_dtype: str                 # "f32" or "bf16"
    grad: str                    # gradient recipe name (see synth.py)
    grad_rank: int = 0           # rank of the structured signal in G
    grad_noise: float = 0.0      # std of the Gaussian noise in G
    grad_signal: float = 0.0     # amplitude of the low-rank signal
    steps: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def elems(self) -> int:
        return sum(s.elems for s in self.mats)


def rank_of(m: int, n: int, rank_div: int) -> int:
    return max(1, min(m, n) // rank_div)


def _spec(name, m, n, r, eta, beta, scale=None):
    return MatrixSpec(name, m, n, r, eta, beta, math.sqrt(m / n) if scale is None else scale)


def single_256x128() -> Workload:
    """One fp32 matrix 256x128, r=16, 10 chained steps, G_t = A_t B_t^T + 0.01 N_t."""
    return Workload(
        "single_256x128_r16", [_spec("w", 256, 128, 16, 0.01, 0.95)], "f32",
        grad="lowrank_plus_noise_host", grad_rank=8, grad_noise=0.01, grad_signal=1.0, steps=10,
        notes="A_t (256x8), B_t (128x8) ~ N(0,1)/sqrt(8); N_t ~ N(0,1); fresh per step from seed 0")


def square_1024(r: int = 256) -> Workload:
    """One 1024x1024 matrix, r=256, bf16 gradient = rank-32 signal + N(0, 0.05^2)."""
    return Workload(
        "square_1024_r256", [_spec("w", 1024, 1024, r, 0.02, 0.95)], "bf16",
        grad="lowrank_plus_noise_host", grad_rank=32, grad_noise=0.05, grad_signal=1.0, steps=10,
        notes="A, B ~ N(0,1)/sqrt(32) (rank 32), noise N(0, 0.05^2), rounded to bf16 (RNE)")


def gpt_160m(rank_div: int = 4) -> Workload:
    """12-layer d=768 GPT: per layer Wq, Wk, Wv, Wo 768x768, up 3072x768, down 768x3072."""
    mats = []
    for layer in range(12):
        for nm, (m, n) in [("q", (768, 768)), ("k", (768, 768)), ("v", (768, 768)),
                           ("o", (768, 768)), ("up", (3072, 768)), ("down", (768, 3072))]:
            mats.append(_spec(f"l{layer}.{nm}", m, n, rank_of(m, n, rank_div), 0.02, 0.95))
    return Workload(f"gpt160m_12L_rdiv{rank_div}", mats, "bf16", grad="lowrank_plus_noise_device",
                    grad_rank=16, grad_noise=1e-3, grad_signal=0.04)


LLAMA3B_SHAPES = [("q", (3072, 3072)), ("k", (1024, 3072)), ("v", (1024, 3072)),
                  ("o", (3072, 3072)), ("gate", (8192, 3072)), ("up", (8192, 3072)),
                  ("down", (3072, 8192))]


def llama_3b(rank_div: int = 16, layers: Optional[List[int]] = None) -> Workload:
    """28-layer Llama-3B (d=3072, GQA 8 KV heads x 128, SwiGLU 8192): 196 matrices."""
    mats = []
    for layer in (range(28) if layers is None else layers):
        for nm, (m, n) in LLAMA3B_SHAPES:
            mats.append(_spec(f"l{layer}.{nm}", m, n, rank_of(m, n, rank_div), 0.02, 0.95))
    return Workload(f"llama3b_28L_rdiv{rank_div}", mats, "bf16", grad="lowrank_plus_noise_device",
                    grad_rank=16, grad_noise=1e-3, grad_signal=0.04)


def sweep(shape=(8192, 8192), r: int = 128) -> Workload:
    """Single-matrix rank sweep: 8192x8192 or 4096x16384, bf16 Gaussian gradient * 1e-3."""
    m, n = shape
    return Workload(f"sweep_{m}x{n}_r{r}", [_spec("w", m, n, r, 0.02, 0.95)], "bf16",
                    grad="gaussian_device", grad_noise=1e-3)


SWEEP_RANKS = [32, 64, 128, 256, 512, 1024, 2048]
SWEEP_SHAPES = [(8192, 8192), (4096, 16384)]


def by_name(name: str) -> Workload:
    table = {
        "single_256x128_r16": single_256x128,
        "square_1024_r256": square_1024,
        "gpt160m_12L_rdiv4": lambda: gpt_160m(4),
        "llama3b_28L_rdiv16": lambda: llama_3b(16),
        "llama3b_28L_rdiv4": lambda: llama_3b(4),
    }
    if name in table:
        return table[name]()
    if name.startswith("sweep_"):
        shp, r = name[len("sweep_"):].split("_r")
        m, n = shp.split("x")
        return sweep((int(m), int(n)), int(r))
    raise KeyError(name)
