"""Float64 CPU oracle for the Dion / Orth-Dion step (test infrastructure only).

Only the tests, the smoke check and the CPU-baseline arm of the bench may
import this package; the library's product path never does.  It is checked
against closed forms, invariants and brute-force SVD cases in
``tests/test_oracle.py`` before it is trusted.
"""
from .dion_oracle import (  # noqa: F401
    DION, ORTH, RANK_TOL, colnorm, default_scale, householder_qr_pos, lapack_qr_pos, orth,
    oracle_chain, oracle_step,
)
