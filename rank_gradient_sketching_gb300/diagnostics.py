"""Gradient-reconstruction diagnostic, composed from the library's kernels.

LoGRA summary page, section "这些节省能说明什么、不能说明什么": the paper
reports the mean cosine similarity between the dense gradient G = dYᵀX of a
micro-batch and its reconstruction R = S·A from the sketch S = G·Aᵀ (about
0.046 at r = 4, 0.348 at r = 256 on real gradients).  For one weight:

    cos(G, R) = ⟨G, R⟩ / (‖G‖·‖R‖),   ⟨G, R⟩ = ⟨G·Aᵀ, S⟩ = ‖S‖².

Every product and norm runs in the library's kernels:
* S by the sketch kernels;
* ‖G‖² without a separate dense GEMM: a sketch whose projection operand is a
  block of `block` unit rows e_j returns (1/√block)·G[:, block columns]
  exactly (P = X·Ãᵀ copies columns of X, so P_lo = 0), so ‖G‖² is block
  times the sum of the squared norms of those sketches;
* R by the merge kernel applied to a zero weight with αη = −1.  R comes out
  rounded to bf16, so each element is within 2⁻⁹ (relative) of S·A and the
  cosine within a factor 1 ± 2⁻⁹ of its exact value.  The errors average out
  over a row only when R takes many distinct values; at r = 4 a row of R
  holds just 8 magnitudes (the sign patterns of 4 ranks), and ‖R‖² moves by
  about 1e-4;
* the norms by `logra_sum_squares` (fp64).
Torch only allocates and fills buffers.  This is a diagnostic: it reads X
and dY k/block + 1 times.
"""

from __future__ import annotations

import math

import torch

from ._binding import (
    logra_merge_update,
    logra_merge_update_proj,
    logra_sketch_accumulate,
    logra_sketch_accumulate_proj,
    logra_sum_squares,
)


def reconstruction_terms(X: torch.Tensor, dY: torch.Tensor, r: int, seed: int = 0, stream_id: int = 0,
                         operand: torch.Tensor | None = None, block: int = 256) -> tuple[float, float, float]:
    """(‖S‖², ‖G‖², ‖S·A‖²) for one micro-batch; A from (seed, stream_id) or a given bf16 operand Ã (r×k)."""
    T, k = X.shape
    d = dY.shape[1]
    dev = X.device
    sums = torch.zeros(3, dtype=torch.float64, device=dev)  # ‖S‖², Σ‖S_b‖², ‖R‖²
    S = torch.zeros((d, r), dtype=torch.float32, device=dev)
    if operand is None:
        logra_sketch_accumulate(X, dY, S, seed, stream_id, r)
    else:
        logra_sketch_accumulate_proj(X, dY, S, operand, r)
    logra_sum_squares(S, sums[0:1])
    sel = torch.zeros((block, k), dtype=torch.bfloat16, device=dev)
    Sb = torch.empty((d, block), dtype=torch.float32, device=dev)
    idx = torch.arange(block, device=dev)
    for b0 in range(0, k, block):
        n = min(block, k - b0)
        sel.zero_()
        sel[idx[:n], b0 + idx[:n]] = 1.0
        Sb.zero_()
        logra_sketch_accumulate_proj(X, dY, Sb, sel, block)
        logra_sum_squares(Sb, sums[1:2], accumulate=True)
    R = torch.zeros((d, k), dtype=torch.bfloat16, device=dev)
    if operand is None:
        logra_merge_update(R, S, seed, stream_id, r, -1.0)
    else:
        logra_merge_update_proj(R, S, operand, r, -1.0)
    logra_sum_squares(R, sums[2:3])
    s2, gb2, r2 = sums.tolist()
    return s2, gb2 * block, r2


def reconstruction_cosine(X: torch.Tensor, dY: torch.Tensor, r: int, seed: int = 0, stream_id: int = 0,
                          operand: torch.Tensor | None = None, block: int = 256) -> float:
    """cos(G, S·A) = ‖S‖²/(‖G‖·‖S·A‖) for one micro-batch (see reconstruction_terms)."""
    s2, g2, r2 = reconstruction_terms(X, dY, r, seed, stream_id, operand, block)
    return s2 / math.sqrt(g2 * r2) if g2 > 0 and r2 > 0 else float("nan")
