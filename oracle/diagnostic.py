"""Gradient-reconstruction diagnostic (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "这些节省能说明什么、不能说明什么": the paper
reports the mean cosine similarity between the dense gradient and its
reconstruction from the sketch, rising from about 0.046 at r = 4 to 0.348 at
r = 256 on real single-micro-batch gradients.  The reconstruction of
G = dYᵀX from its sketch S = G·Aᵀ is R = S·A (the same product the merge
applies), so the diagnostic of one weight and micro-batch is

    cos(G, R) = ⟨G, R⟩ / (‖G‖_F · ‖R‖_F).

Written out here with G formed explicitly in fp64.

Pinned by (tests/test_oracle.py): an orthonormal A (AAᵀ = I) whose row space
contains the rows of G reconstructs G exactly (cos = 1); for a random G the
value approaches tr(AAᵀ)/√(k·‖AAᵀ‖_F²), which for random signs is close to
√(r/(r + k)); invariance to the scale of X and of dY; and ⟨G, R⟩ = ‖S‖_F².
"""

from __future__ import annotations

import numpy as np


def reconstruction_cosine(X: np.ndarray, dY: np.ndarray, A: np.ndarray) -> float:
    """cos(G, S·A) for one micro-batch (X T×k, dY T×d, A r×k)."""
    G = np.asarray(dY, dtype=np.float64).T @ np.asarray(X, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    R = (G @ A.T) @ A
    return float(np.sum(G * R) / (np.linalg.norm(G) * np.linalg.norm(R)))
