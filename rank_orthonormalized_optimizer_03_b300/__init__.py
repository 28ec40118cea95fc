"""Dion / Orth-Dion optimizer step for NVIDIA B300 (sm_103a).

The step itself runs in hand-written CUDA kernels behind a C ABI
(``libdion.so``, declared in ``include/dion.h``); this package is a thin
ctypes binding over it plus the workload definitions and the seeded input
generators.
"""
from . import workloads, synth  # noqa: F401
