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
path stays in the library's kernels.  The policy-sync payload at the end of
this module is what a trainer sends a rollout replica after a step.
"""

from __future__ import annotations

import contextlib

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


# ----------------------------------------------------------------------------
# Policy-sync payload (section "同一份草图也压缩策略同步开销"): the receiving side
# regenerates A from the seed and applies the received factor; what travels is
# U = S (d·r fp32 numbers), αη, the seed and the stream id of each sketched
# weight — never a d×k update.
#
# Layout (little-endian):
#   file header  : magic b"LGRP", version u16, count u32
#   per entry    : name length u16, name (utf-8), d i64, k i64, r i32,
#                  seed u64, stream_id u32, alpha_eta f64,
#                  then d·r fp32 values of S, row-major
# ----------------------------------------------------------------------------
import struct  # noqa: E402

_MAGIC = b"LGRP"
_VERSION = 1
_ENTRY = struct.Struct("<qqiQId")


def sync_payload_bytes(shapes) -> int:
    """Size in bytes of a payload for [(name, d, r)]; O(Σ d·r), independent of k."""
    total = 4 + 2 + 4
    for name, d, r in shapes:
        total += 2 + len(name.encode()) + _ENTRY.size + 4 * d * r
    return total


def pack_sync_payload(entries) -> bytes:
    """entries: [(name, S (d×r fp32 tensor, any device), k, seed, stream_id, alpha_eta)]."""
    parts = [_MAGIC, struct.pack("<HI", _VERSION, len(entries))]
    for name, S, k, seed, sid, alpha_eta in entries:
        if S.dtype != torch.float32 or S.dim() != 2:
            raise TypeError("S must be a 2-D float32 tensor")
        nb = name.encode()
        d, r = S.shape
        parts.append(struct.pack("<H", len(nb)) + nb + _ENTRY.pack(d, int(k), r, int(seed), int(sid),
                                                                      float(alpha_eta)))
        parts.append(S.detach().to("cpu").contiguous().numpy().astype("<f4", copy=False).tobytes())
    return b"".join(parts)


def unpack_sync_payload(payload: bytes):
    """[(name, S (cpu fp32), k, seed, stream_id, alpha_eta)] from pack_sync_payload's bytes."""
    import numpy as np

    mv = memoryview(payload)
    if bytes(mv[:4]) != _MAGIC:
        raise ValueError("not a sketch sync payload")
    version, count = struct.unpack_from("<HI", mv, 4)
    if version != _VERSION:
        raise ValueError(f"unsupported payload version {version}")
    off, out = 10, []
    for _ in range(count):
        (nlen,) = struct.unpack_from("<H", mv, off)
        off += 2
        name = bytes(mv[off:off + nlen]).decode()
        off += nlen
        d, k, r, seed, sid, ae = _ENTRY.unpack_from(mv, off)
        off += _ENTRY.size
        S = torch.from_numpy(np.frombuffer(payload, dtype="<f4", count=d * r, offset=off).reshape(d, r).copy())
        off += 4 * d * r
        out.append((name, S, k, seed, sid, ae))
    if off != len(payload):
        raise ValueError("trailing bytes in payload")
    return out


def _byte_range(W: torch.Tensor) -> tuple[int, int]:
    """[first, last + 1) byte addresses of a 2-D row-major tensor's elements."""
    d, k = W.shape
    n = (d - 1) * W.stride(0) + k if d and k else 0
    return W.data_ptr(), W.data_ptr() + n * W.element_size()


def _overlaps(a: tuple[int, int], ranges) -> bool:
    return any(a[0] < b[1] and b[0] < a[1] for b in ranges)


def apply_sync_payload(payload: bytes, weights, stream=None, grouped: bool = True) -> None:
    """Applies W ← bf16(W − αη·U·A) for every entry to weights[name] (bf16 d×k
    device tensors), A regenerated from the entry's seed and stream id.

    Everything (the copies of S to the device, the plans, the merges) is
    enqueued on `stream` (default: the current stream), so the buffers it
    allocates are only reused by work ordered after the merges.

    grouped: entries are merged in batches, one launch per batch over a plan
    (logra_merge_update_group).  A batch holds entries of one (r, αη) whose
    weights do not overlap in memory; an entry whose weight overlaps one
    already batched (a name given twice, or two names for one tensor, as with
    tied weights) starts a new batch that runs after it.  So the weights end
    bit-identical to one merge per entry in payload order (grouped=False)."""
    from ._binding import logra_merge_group_plan, logra_merge_update, logra_merge_update_group

    entries = unpack_sync_payload(payload)
    for name, S, k, seed, sid, ae in entries:
        W = weights[name]
        if W.shape[0] != S.shape[0] or W.shape[1] != k:
            raise ValueError(f"{name}: payload is {S.shape[0]}×{k}, weight is {tuple(W.shape)}")
    if not entries:
        return
    dev = weights[entries[0][0]].device
    if dev.type == "cuda":
        st = stream if isinstance(stream, torch.cuda.Stream) else (
            torch.cuda.ExternalStream(stream, device=dev) if stream is not None else torch.cuda.current_stream(dev))
        ctx = torch.cuda.stream(st)
    else:  # host tensors: only the batching logic runs (tests with a stand-in binding)
        st, ctx = stream, contextlib.nullcontext()
    with ctx:
        # batches in launch order: [key, targets, byte ranges]
        batches = []
        for name, S, k, seed, sid, ae in entries:
            W = weights[name]
            S_dev = S.to(W.device, non_blocking=False)
            if not grouped:
                logra_merge_update(W, S_dev, seed, sid, S.shape[1], ae, stream=st)
                continue
            key, rng = (S.shape[1], ae), _byte_range(W)
            # the newest batch of this key, if no batch from it onwards holds an overlapping weight
            last = max((i for i, b in enumerate(batches) if b[0] == key), default=None)
            if last is None or any(_overlaps(rng, b[2]) for b in batches[last:]):
                batches.append([key, [], []])
                last = len(batches) - 1
            batches[last][1].append((W, S_dev, seed, sid))
            batches[last][2].append(rng)
        for (r, ae), targets, _ in batches:
            plan = logra_merge_group_plan(targets, r, stream=st)
            logra_merge_update_group(plan, ae, stream=st)


def broadcast_sync_payload(payload: bytes | None, src: int = 0, group=None) -> bytes:
    """Sends the payload from rank src to every rank (torch.distributed)."""
    n = torch.tensor([len(payload) if payload is not None else 0], dtype=torch.int64)
    dist.broadcast(n, src, group=group)
    buf = torch.empty(int(n.item()), dtype=torch.uint8)
    if dist.get_rank(group) == src:
        buf.copy_(torch.frombuffer(bytearray(payload), dtype=torch.uint8))
    dist.broadcast(buf, src, group=group)
    return buf.numpy().tobytes()
