"""Momentum on the sketch (oracle side) — a reading, not a rule of the pages.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "草图如何取代完整梯度缓冲": the plain update uses
U = S, and a stateful sketch optimiser is mentioned only as something that
adds storage of its own; no rule is given.  The reading implemented here is
heavy-ball momentum kept on the d×r sketch itself:

    M_t = β·M_{t−1} + S_t,      U_t = M_t,      W ← W − αη·U_t·A

with M_0 = 0.  It needs a fixed projection (the same seed and stream id every
step), so that every S_t, and hence M_t, lives in the same r-dimensional
basis.  β is taken at the precision the caller passes it in (fp32 on the
device side), widened exactly to fp64 here.

Pinned by (tests/test_oracle.py): β = 0 gives M = S exactly; a constant S
gives the geometric-series closed form S·(1 − βⁿ)/(1 − β) after n steps; β = 1
gives the plain sum of the sketches; linearity in (M, S); and, with the merge
oracle, that U = M_t applied through one merge equals the same update
written out from its closed form.
"""

from __future__ import annotations

import numpy as np


def momentum_update(M: np.ndarray, S: np.ndarray, beta: float) -> np.ndarray:
    """One step of M ← β·M + S in fp64 (returns the new M)."""
    M = np.asarray(M, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    if M.shape != S.shape:
        raise ValueError("M and S must have the same shape")
    return float(beta) * M + S


def momentum_run(sketches, beta: float) -> np.ndarray:
    """M_n after feeding the sketches S_1..S_n in order, starting from M_0 = 0."""
    M = None
    for S in sketches:
        M = np.zeros_like(np.asarray(S, dtype=np.float64)) if M is None else M
        M = momentum_update(M, S, beta)
    if M is None:
        raise ValueError("no sketches")
    return M
