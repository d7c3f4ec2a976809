"""Merge update W′ = bf16(W − αη·U·A) with U = S (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "草图如何取代完整梯度缓冲": the update has the form
W ← W − αηUA, with U = S in the basic SGD variant, merged straight into the
weights with no resident adapter branch.  The pages state no rounding mode for
the bf16 weights; the reading taken here is round-to-nearest-even of the exact
fp64 result, done in one step (no intermediate fp32 rounding).

Pinned by: αη = 0 leaving W bit-for-bit unchanged, the closed form for a
single non-zero entry of S, and ``bf16_round`` against hand-worked ties and
against PyTorch's fp32→bf16 conversion on fp32-representable inputs.
"""

from __future__ import annotations

import numpy as np

_BF16_MANT = 8  # significant bits, hidden bit included
_BF16_EMIN = -126  # smallest normal exponent
_BF16_MAX = float.fromhex("0x1.fe00000000000p+127")


def bf16_round(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as
    fp64.  Handles subnormals, overflow to ±inf, NaN and signed zero."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    m, e = np.frexp(xf)  # xf = m·2^e, 0.5 ≤ |m| < 1
    # Value of one unit in the last place for each input: 2^(e-8) for normals,
    # and the fixed subnormal spacing 2^-133 below the normal range.
    exp_ulp = np.maximum(e - _BF16_MANT, _BF16_EMIN - (_BF16_MANT - 1))
    q = np.rint(np.ldexp(xf, -exp_ulp))  # np.rint rounds half to even
    y = np.ldexp(q, exp_ulp)
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, xf), y)
    y = np.where(y == 0, np.copysign(0.0, xf), y)
    out[finite] = y
    return out


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (the ulp of the binade containing x)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x == 0, 1e-300, x))
    exp_ulp = np.maximum(e - _BF16_MANT, _BF16_EMIN - (_BF16_MANT - 1))
    return np.ldexp(1.0, exp_ulp)


def update(S: np.ndarray, A: np.ndarray, alpha_eta: float) -> np.ndarray:
    """The exact fp64 update αη·S·A (d×k)."""
    return float(alpha_eta) * (np.asarray(S, dtype=np.float64) @ np.asarray(A, dtype=np.float64))


def merge(W: np.ndarray, S: np.ndarray, A: np.ndarray, alpha_eta: float) -> np.ndarray:
    """bf16_rne(W − αη·S·A) as fp64 values (W holds bf16 values widened)."""
    W = np.asarray(W, dtype=np.float64)
    return bf16_round(W - update(S, A, alpha_eta))
