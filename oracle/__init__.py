"""Float64 CPU oracle for the Matryoshka contrastive losses (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` /
``--impl reference`` leg may import this package.  The CUDA library never calls it,
and the two share no code: this package wraps ``oracle.c`` (plain C, float64,
OpenMP) through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, torch library routines, autograd, finite differences, invariants).
"""
from .ref import (  # noqa: F401
    KINDS,
    build,
    fwd_bwd,
    row_stats,
    softmax_normalisers,
    row_terms_sampled,
    grad_rows,
    scale_grads,
    label_matrix,
    oneset,
)
