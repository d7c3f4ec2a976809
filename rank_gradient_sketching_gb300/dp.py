"""Data-parallel exchange of the sketching hot path (host side).

LoGRA summary page, section "同一份草图也压缩策略同步开销": what ranks exchange
is the compact sketch (O(d·r) numbers) plus the projection seed, never a d×k
update.  With micro-batches spread over ranks, S is linear in the micro-batches
(section "草图如何取代完整梯度缓冲": each micro-batch's projected contribution is
added into S), so the step's sketch is the sum of the ranks' sketches: one
all-reduce of the flat sketch buffer before the merge.  The predicted KL is a
mean over token rows, so the global q(D) is the row-weighted mean of the ranks'
values.  Every rank then applies the same merge (same S, same seed).

These helpers only move data with torch.distributed; the arithmetic of the
path stays in the library's kernels.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def allreduce_sketch(s_flat: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the flat fp32 sketch buffer over the ranks, in place."""
    if s_flat.dtype != torch.float32:
        raise TypeError("sketch buffer must be float32")
    dist.all_reduce(s_flat, op=dist.ReduceOp.SUM, group=group)
    return s_flat


def global_q(q_local: torch.Tensor, rows_local: int, group=None) -> torch.Tensor:
    """Row-weighted mean of the ranks' q(D), in place in q_local (fp64 scalar).

    A rank with no selected rows contributes nothing; with no rows anywhere
    the result is 0, matching the single-rank convention."""
    if q_local.dtype != torch.float64:
        raise TypeError("q must be float64")
    buf = torch.stack([q_local.reshape(()) * rows_local,
                       torch.tensor(float(rows_local), dtype=torch.float64, device=q_local.device)])
    dist.all_reduce(buf, op=dist.ReduceOp.SUM, group=group)
    total_rows = buf[1]
    q_local.copy_(torch.where(total_rows > 0, buf[0] / total_rows.clamp(min=1.0), torch.zeros_like(buf[0])))
    return q_local
