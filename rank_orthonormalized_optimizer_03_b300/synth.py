"""Seeded synthetic inputs for the Dion / Orth-Dion step.

This module only draws random numbers and rounds them to the storage types;
it holds none of the method's arithmetic.  Both the CUDA path (tests, bench)
and the float64 oracle (tests) take their inputs from here, so the two sides
always see identical stored values.

Recipes (per matrix, in draw order):

* ``X0``      ~ N(0, 0.02^2), stored fp32.
* ``V0_raw``  ~ N(0, 1), n x r.  The warm start V_0 is orth(V0_raw); the
  orthonormalisation is done by whichever side consumes it (it is the
  method's own orth), never here.
* ``R0``      = 0.
* ``G``       = signal * A B^T + noise * N, with A (m x k), B (n x k)
  ~ N(0, 1)/sqrt(k) and N ~ N(0, 1); rounded to fp32 and then, for a bf16
  gradient, to bf16 with round-to-nearest-even.

Host workloads (single matrices) draw from ``numpy.random.PCG64(seed)``;
device workloads (batched models, sweeps) from ``torch.Generator`` seeded
per matrix with ``seed * 1_000_003 + index`` on the target device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

from .workloads import MatrixSpec, Workload


# ---------------------------------------------------------------- bf16 bits
def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).astype(np.uint32) << 16
    return b.view(np.float32)


# ---------------------------------------------------------------- host draws
@dataclass
class HostInputs:
    """Inputs of one single-matrix workload, as stored (fp32 / bf16 bits)."""
    spec: MatrixSpec
    X0: np.ndarray                 # m x n float32
    V0_raw: np.ndarray             # n x r float64 (orthonormalised by the consumer)
    grads: List[np.ndarray]        # per step: m x n float32, or uint16 bf16 bits
    g_dtype: str

    def grad_f64(self, t: int) -> np.ndarray:
        g = self.grads[t]
        if self.g_dtype == "bf16":
            return bf16_bits_to_f32(g).astype(np.float64)
        return g.astype(np.float64)


def host_inputs(wl: Workload, seed: int = 0, steps: Optional[int] = None) -> HostInputs:
    """Draw the inputs of a single-matrix workload on the host (PCG64)."""
    if len(wl.mats) != 1:
        raise ValueError("host_inputs covers single-matrix workloads")
    spec = wl.mats[0]
    m, n, r = spec.m, spec.n, spec.r
    steps = wl.steps if steps is None else steps
    rng = np.random.Generator(np.random.PCG64(seed))
    X0 = rng.normal(0.0, 0.02, size=(m, n)).astype(np.float32)
    V0_raw = rng.standard_normal((n, r))
    grads = []
    for _ in range(steps):
        grads.append(_draw_grad_host(rng, wl, m, n))
    return HostInputs(spec, X0, V0_raw, grads, wl.g_dtype)


def _draw_grad_host(rng, wl: Workload, m: int, n: int) -> np.ndarray:
    if wl.grad == "lowrank_plus_noise_host":
        k = wl.grad_rank
        A = rng.standard_normal((m, k)) / math.sqrt(k)
        B = rng.standard_normal((n, k)) / math.sqrt(k)
        N = rng.standard_normal((m, n))
        g = (wl.grad_signal * (A @ B.T) + wl.grad_noise * N).astype(np.float32)
    elif wl.grad in ("gaussian_host", "gaussian_device"):
        g = (wl.grad_noise * rng.standard_normal((m, n))).astype(np.float32)
    elif wl.grad == "lowrank_plus_noise_device":
        k = wl.grad_rank
        A = rng.standard_normal((m, k)) / math.sqrt(k)
        B = rng.standard_normal((n, k)) / math.sqrt(k)
        N = rng.standard_normal((m, n))
        g = (wl.grad_signal * (A @ B.T) + wl.grad_noise * N).astype(np.float32)
    else:
        raise ValueError(wl.grad)
    return f32_to_bf16_bits(g) if wl.g_dtype == "bf16" else g


def host_matrix_inputs(spec: MatrixSpec, wl: Workload, seed: int):
    """Host draw of one matrix of a batched workload (used for CPU-side samples)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    X0 = rng.normal(0.0, 0.02, size=(spec.m, spec.n)).astype(np.float32)
    V0_raw = rng.standard_normal((spec.n, spec.r))
    G = _draw_grad_host(rng, wl, spec.m, spec.n)
    return X0, V0_raw, G


# ---------------------------------------------------------------- device draws
def device_matrix_inputs(spec: MatrixSpec, wl: Workload, index: int, seed: int = 0,
                         device="cuda"):
    """Draw (X0, V0_raw, G) for matrix ``index`` of a batched workload with torch.

    X0 float32 m x n, V0_raw float32 n x r (to be orthonormalised by the
    consumer), G bf16 (or float32) m x n, all on ``device``.
    """
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + index)
    m, n, r = spec.m, spec.n, spec.r
    X0 = torch.randn((m, n), generator=gen, device=device, dtype=torch.float32) * 0.02
    V0_raw = torch.randn((n, r), generator=gen, device=device, dtype=torch.float32)
    N = torch.randn((m, n), generator=gen, device=device, dtype=torch.float32)
    if wl.grad == "lowrank_plus_noise_device":
        k = wl.grad_rank
        A = torch.randn((m, k), generator=gen, device=device, dtype=torch.float32) / math.sqrt(k)
        B = torch.randn((n, k), generator=gen, device=device, dtype=torch.float32) / math.sqrt(k)
        G = N.mul_(wl.grad_noise).addmm_(A, B.t(), alpha=wl.grad_signal)
    elif wl.grad == "gaussian_device":
        G = N.mul_(wl.grad_noise)
    else:
        raise ValueError(wl.grad)
    G = G.to(torch.bfloat16) if wl.g_dtype == "bf16" else G
    return X0, V0_raw, G
