"""Predicted KL q(D) between the current and the proposed model (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "预测 KL 控制防止过大更新破坏学习": a small set of
sampled responses is taken from the batch and the vocabulary distribution of
the current model is compared with that of the proposed (updated) model at the
same temperature; the mean predicted KL is q(D).

Readings (the pages leave them open): the divergence is KL(current ‖
proposed) = Σ_v p_v (log p_v − log p′_v) with p = softmax(a/τ) from the
current logits a and p′ = softmax(b/τ) from the proposed logits b; q(D) is the
plain mean over the selected token rows.  Terms with p_v = 0 contribute 0; a
finite a_v with b_v = −inf gives +inf; NaN propagates.

This is the plain definition in fp64 (max-subtracted log-softmax).

Pinned by: KL ≥ 0 and = 0 exactly for b = a, the two-token closed form, the
uniform-logit closed form, scipy.special.rel_entr, and the page's quadratic
model (the KL of a + αΔ scales as α² for small α).
"""

from __future__ import annotations

import numpy as np


def log_softmax(z: np.ndarray) -> np.ndarray:
    """Row-wise log-softmax in fp64 (rows along the last axis)."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        lse = m + np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True))
    return z - lse


def token_kl(cur: np.ndarray, prop: np.ndarray, temperature: float) -> np.ndarray:
    """Per-row KL(softmax(cur/τ) ‖ softmax(prop/τ)) in fp64, shape (rows,)."""
    if not temperature > 0:
        raise ValueError("temperature must be > 0")
    lp = log_softmax(np.asarray(cur, dtype=np.float64) / temperature)
    lq = log_softmax(np.asarray(prop, dtype=np.float64) / temperature)
    p = np.exp(lp)
    with np.errstate(invalid="ignore"):
        terms = np.where(p == 0, 0.0, p * (lp - lq))
    # NaN inputs must surface even where p underflowed to 0.
    nan_rows = np.isnan(np.asarray(cur, dtype=np.float64)).any(-1) | np.isnan(
        np.asarray(prop, dtype=np.float64)
    ).any(-1)
    out = np.sum(terms, axis=-1)
    out[nan_rows] = np.nan
    return out


def predicted_kl(cur, prop, temperature: float, row_mask=None) -> tuple[float, np.ndarray]:
    """(q(D), per-row KL).  q(D) is the mean over rows whose mask is non-zero
    (all rows when row_mask is None); with no selected rows q(D) = 0."""
    kl = token_kl(cur, prop, temperature)
    if row_mask is None:
        sel = kl
    else:
        sel = kl[np.asarray(row_mask).astype(bool)]
    q = float(np.mean(sel)) if sel.size else 0.0
    return q, kl
