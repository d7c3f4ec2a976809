"""Philox4x32-10 and the Rademacher projection A (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The projection: LoGRA summary page, section "草图如何取代完整梯度缓冲" — A is
r×k, drawn independently of the batch, fixed during accumulation, not
learned; by default its entries are independent random signs scaled by 1/√r.
Section "同一份草图也压缩策略同步开销" — the rollout side regenerates A from a
seed, so A is a pure function of (seed, matrix identity).

The pages name no generator.  Reading taken here (and on the CUDA side,
independently written): Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11,
"Parallel random numbers: as easy as 1, 2, 3", section 3.2, with the
multipliers and Weyl key increments given there) with

    key     = (seed mod 2³², seed >> 32)
    counter = (j >> 7, i, stream_id, 0)        for row i, column j of A
    bit     = (word[(j & 127) >> 5] >> (j & 31)) & 1
    sign    = −1 if bit else +1

so one Philox call yields 128 consecutive columns of one row.

Pinned by: the Random123 known-answer vectors (tests/golden/), the exact
diagonal of AᵀA, sign balance, and (on a GPU) cuRAND's device Philox4x32-10.
"""

from __future__ import annotations

import numpy as np

# Philox4x32 round multipliers and key increments (SC'11, section 3.2).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9  # golden ratio
PHILOX_W1 = 0xBB67AE85  # sqrt(3) - 1
MASK32 = 0xFFFFFFFF


def _mulhilo(a: np.ndarray, m: int) -> tuple[np.ndarray, np.ndarray]:
    """Full 64-bit product of two 32-bit words, split into (hi, lo)."""
    p = a.astype(np.uint64) * np.uint64(m)
    return (p >> np.uint64(32)).astype(np.uint32), (p & np.uint64(MASK32)).astype(np.uint32)


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32 with 10 rounds.

    counter: array-like (..., 4) of uint32; key: array-like (..., 2) of uint32
    (broadcast against each other).  Returns (..., 4) uint32.

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1·c2) ⊕ c1 ⊕ k0, lo(M1·c2), hi(M0·c0) ⊕ c3 ⊕ k1, lo(M0·c0));
    the key is bumped by (W0, W1) between rounds.
    """
    ctr = np.asarray(counter, dtype=np.uint64)
    k = np.asarray(key, dtype=np.uint64)
    parts = np.broadcast_arrays(ctr[..., 0], ctr[..., 1], ctr[..., 2], ctr[..., 3], k[..., 0], k[..., 1])
    c0, c1, c2, c3 = (p.astype(np.uint32) for p in parts[:4])
    k0, k1 = (p.astype(np.uint64) & MASK32 for p in parts[4:])
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        hi0, lo0 = _mulhilo(c0, PHILOX_M0)
        hi1, lo1 = _mulhilo(c2, PHILOX_M1)
        c0, c1, c2, c3 = (
            hi1 ^ c1 ^ k0.astype(np.uint32),
            lo1,
            hi0 ^ c3 ^ k1.astype(np.uint32),
            lo0,
        )
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def sign_bits(seed: int, stream_id: int, r: int, k: int) -> np.ndarray:
    """Raw sign bits of A as a uint8 array (r, k); 1 means −1."""
    if r < 0 or k < 0:
        raise ValueError("r and k must be non-negative")
    groups = (k + 127) // 128
    i = np.arange(r, dtype=np.uint64)[:, None]
    g = np.arange(groups, dtype=np.uint64)[None, :]
    ctr = np.zeros((r, groups, 4), dtype=np.uint64)
    ctr[..., 0] = g
    ctr[..., 1] = i
    ctr[..., 2] = np.uint64(stream_id & MASK32)
    key = np.array([seed & MASK32, (seed >> 32) & MASK32], dtype=np.uint64)
    words = philox4x32_10(ctr, np.broadcast_to(key, (r, groups, 2)))  # (r, groups, 4)
    j = np.arange(k)
    w = words[:, j >> 7, (j & 127) >> 5]  # (r, k)
    return ((w >> (j & 31).astype(np.uint32)) & 1).astype(np.uint8)


def signs(seed: int, stream_id: int, r: int, k: int) -> np.ndarray:
    """A·√r as int8 ±1, shape (r, k)."""
    return (1 - 2 * sign_bits(seed, stream_id, r, k).astype(np.int16)).astype(np.int8)


def projection(seed: int, stream_id: int, r: int, k: int) -> np.ndarray:
    """The projection A itself in fp64: entries ±1/√r, shape (r, k)."""
    return signs(seed, stream_id, r, k).astype(np.float64) / np.sqrt(r)


# ---------------------------------------------------------------------------
# Refreshed basis.  Summary page, section "这些节省能说明什么、不能说明什么"
# (the design-choice experiments): besides a fixed Rademacher basis the paper
# runs refreshed Rademacher and refreshed Gaussian projections, i.e. A is
# redrawn every step.  The pages do not say how the new draw is keyed.  Reading
# taken here: step t uses the 64-bit seed
#
#     seed_t = w0 | (w1 << 32),   (w0, w1, ·, ·) = Philox4x32-10(
#                                     counter = (t mod 2³², t >> 32, 0, 2),
#                                     key     = (base mod 2³², base >> 32))
#
# so that consecutive steps get unrelated keys.  The fourth counter word keeps
# this use of the generator apart from the signs (0) and the Gaussian draws (1).
# ---------------------------------------------------------------------------
def refreshed_seed(base_seed: int, step: int) -> int:
    if step < 0:
        raise ValueError("step must be >= 0")
    ctr = np.array([step & MASK32, (step >> 32) & MASK32, 0, 2], dtype=np.uint64)
    key = np.array([base_seed & MASK32, (base_seed >> 32) & MASK32], dtype=np.uint64)
    w = philox4x32_10(ctr, key)
    return int(w[0]) | (int(w[1]) << 32)
