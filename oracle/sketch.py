"""Sketch accumulation S = Σ_m G_m Aᵀ, with G_m = dY_mᵀ X_m formed explicitly.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "草图如何取代完整梯度缓冲": for a d×k weight W the
method keeps the d×r sketch S = G Aᵀ instead of the d×k gradient G, adding
each micro-batch's projected contribution into S in fp32.  For a linear layer
y = W x the weight gradient of one micro-batch is G = dYᵀ X (T tokens, X is
T×k, dY is T×d) — the outer-product form ∂L/∂W = Σ_t ∂L/∂y_t · x_tᵀ.

This module deliberately takes the *unoptimised* route the method avoids: it
forms G in fp64 and multiplies by the materialised A.  Inputs are the exact
bf16 values widened to fp64.

Pinned by: brute-force loops of the projected-input form dYᵀ(X Aᵀ) on tiny
shapes, linearity across micro-batches, and the page's d=k=4096, r=64 memory
arithmetic (64 MiB versus 1 MiB).
"""

from __future__ import annotations

import numpy as np


def dense_gradient(X: np.ndarray, dY: np.ndarray) -> np.ndarray:
    """G = dYᵀ X (d×k) in fp64 for one micro-batch (X: T×k, dY: T×d)."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    if X.ndim != 2 or dY.ndim != 2 or X.shape[0] != dY.shape[0]:
        raise ValueError("X is T×k and dY is T×d with the same T")
    return dY.T @ X


def sketch_accumulate(S0: np.ndarray, microbatches, A: np.ndarray) -> np.ndarray:
    """S0 + Σ_m (dY_mᵀ X_m) Aᵀ in fp64.

    S0: d×r initial sketch; microbatches: iterable of (X_m, dY_m); A: r×k.
    """
    S = np.array(S0, dtype=np.float64, copy=True)
    A = np.asarray(A, dtype=np.float64)
    for X, dY in microbatches:
        G = dense_gradient(X, dY)
        if G.shape[1] != A.shape[1] or G.shape[0] != S.shape[0] or A.shape[0] != S.shape[1]:
            raise ValueError("shape mismatch between G (d×k), A (r×k) and S (d×r)")
        S += G @ A.T
    return S


def sketch_rows(S0_rows: np.ndarray, rows, microbatches, A: np.ndarray) -> np.ndarray:
    """The same sum restricted to a set of output rows of S (for large shapes).

    Row i of G is dY[:, i]ᵀ X, so only those rows of the dense gradient are
    formed.
    """
    rows = np.asarray(rows)
    S = np.array(S0_rows, dtype=np.float64, copy=True)
    A = np.asarray(A, dtype=np.float64)
    for X, dY in microbatches:
        X = np.asarray(X, dtype=np.float64)
        dYr = np.asarray(dY, dtype=np.float64)[:, rows]
        G_rows = dYr.T @ X
        S += G_rows @ A.T
    return S


def accumulator_bytes(d: int, k: int, r: int, itemsize: int = 4) -> tuple[int, int]:
    """(bytes of a d×k gradient accumulator, bytes of the d×r sketch) at the
    given element size; the page's example is d = k = 4096, r = 64, fp32."""
    return d * k * itemsize, d * r * itemsize
