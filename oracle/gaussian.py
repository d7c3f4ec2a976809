"""Gaussian projection (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "这些节省能说明什么、不能说明什么" (design-choice
experiments): the paper compares fixed Rademacher, refreshed Rademacher and
refreshed Gaussian projections.  The pages give neither the generator nor
the transform.  Readings taken here (the CUDA side is written independently
from the same definition):

* Normals by the Box–Muller transform (Box and Muller, "A note on the
  generation of random normal deviates", Ann. Math. Stat. 29, 1958) from
  Philox4x32-10 words: for row i and columns 4q .. 4q+3 of A

      (w0, w1, w2, w3) = Philox4x32-10(counter = (q, i, stream_id, 1),
                                       key = (seed mod 2³², seed >> 32))
      u = (w0 + ½)·2⁻³²,  φ = (w1 + ½)·2⁻³²       (both in (0, 1))
      z[4q]   = √(−2 ln u)·cos 2πφ,   z[4q+1] = √(−2 ln u)·sin 2πφ
      z[4q+2], z[4q+3] the same from (w2, w3).

* The projection operand is Ã = bf16_rn(z) and A = Ã/√r, so that
  E[AᵀA] = I as for the signs.  The rounding to bf16 is part of the
  definition: the tensor cores take A as bf16, and an fp32 A would leave the
  sketch about 1.1e-3 (relative Frobenius) away from one built with bf16
  entries, above the 1e-3 bound.

Pinned by (tests/test_oracle.py): a Kolmogorov–Smirnov test of z against the
standard normal CDF, the first four moments, zero correlation between the
two outputs of one pair and between neighbouring columns, E[AᵀA] ≈ I, and
the symmetry z ↦ −z of the distribution; the bf16 rounding is the merge
oracle's, pinned on its own.
"""

from __future__ import annotations

import numpy as np

from .merge import bf16_round
from .philox import MASK32, philox4x32_10


def normals(seed: int, stream_id: int, r: int, k: int) -> np.ndarray:
    """z in fp64, shape (r, k)."""
    if r < 0 or k < 0:
        raise ValueError("r and k must be non-negative")
    quads = (k + 3) // 4
    ctr = np.zeros((r, quads, 4), dtype=np.uint64)
    ctr[..., 0] = np.arange(quads, dtype=np.uint64)[None, :]
    ctr[..., 1] = np.arange(r, dtype=np.uint64)[:, None]
    ctr[..., 2] = np.uint64(stream_id & MASK32)
    ctr[..., 3] = 1
    key = np.array([seed & MASK32, (seed >> 32) & MASK32], dtype=np.uint64)
    w = philox4x32_10(ctr, np.broadcast_to(key, (r, quads, 2))).astype(np.float64)
    u = (w[..., 0::2] + 0.5) * 2.0**-32      # (r, quads, 2): u of each pair
    phi = (w[..., 1::2] + 0.5) * 2.0**-32
    rho = np.sqrt(-2.0 * np.log(u))
    z = np.empty((r, quads, 4))
    z[..., 0::2] = rho * np.cos(2.0 * np.pi * phi)
    z[..., 1::2] = rho * np.sin(2.0 * np.pi * phi)
    return z.reshape(r, quads * 4)[:, :k]


def operand(seed: int, stream_id: int, r: int, k: int) -> np.ndarray:
    """Ã = bf16_rn(z) (values in fp64), the tensor-core operand."""
    return bf16_round(normals(seed, stream_id, r, k))


def projection(seed: int, stream_id: int, r: int, k: int) -> np.ndarray:
    """A = Ã/√r in fp64, shape (r, k)."""
    return operand(seed, stream_id, r, k) / np.sqrt(r)
