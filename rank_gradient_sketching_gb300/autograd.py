"""Backward-pass integration: linear layers whose weight gradient is never formed.

LoGRA summary page, section "草图如何取代完整梯度缓冲": the compressed weight
matrices never get a full gradient buffer — each micro-batch's contribution is
projected and added into the sketch S during the backward pass, and the update
W ← W − αηUA (U = S) is merged straight into the weights.  Section
"这些节省能说明什么、不能说明什么" and the evaluation page: the sketched
matrices are the attention and feed-forward projections; other parameters
follow their usual path.

`SketchedLinearGroup` holds one or more bf16 weights that read the same input
(a layer's q/k/v, or gate/up, or a single projection).  Its backward returns
the input gradient Σ_j dY_j W_j (a library GEMM: it belongs to the model's own
backward, not to the sketch) and, in place of dW_j = dY_jᵀX, adds the
projected contribution into each S_j: at once through
`logra_sketch_accumulate_shared_x`, which reads X once for the whole group,
or, inside a `SketchBatch` context, deferred and run for the weights of many
groups together by `logra_sketch_accumulate_group` (one launch per phase,
which fills the GPU from one stream where a single group's call would not).
`merge_` applies W_j ← W_j − αη·S_j·A_j and clears S_j.  `GroupMerger` does
the same for the weights of many groups (a whole model's sketched
projections) in one launch over a plan (`logra_merge_update_group`).
"""

from __future__ import annotations

import torch

from ._binding import (
    LOGRA_MAX_SHARED_X_TARGETS,
    _torch_stream,
    logra_merge_group_plan,
    logra_merge_update,
    logra_merge_update_group,
    logra_merge_update_proj,
    logra_sketch_accumulate_group,
    logra_sketch_accumulate_shared_x,
    logra_sketch_accumulate_shared_x_proj,
    logra_sketch_group_plan,
    logra_sketch_group_workspace_bytes,
    logra_sketch_shared_x_workspace_bytes,
)

# The batches whose context is open, innermost last.  Process-wide, not per
# thread: the autograd engine runs the backward of CUDA tensors on a worker
# thread of its own.  So one thread at a time runs a backward into a batch.
_active_batches = []


def _current_batch():
    return _active_batches[-1] if _active_batches else None


class SketchBatch:
    """Defers the sketch work of `SketchedLinearGroup` backward passes and runs
    it as grouped launches (`logra_sketch_accumulate_group`):

        with SketchBatch():
            loss.backward()

    Each backward inside the context hands its (X, dY, S, projection) targets
    to the batch instead of launching.  The batch runs what it holds when the
    inputs it holds reach `flush_bytes`, before it
    would take a second contribution to an S it already holds (a group used
    twice in one graph), and when the context ends without an exception; the
    input and output tensors stay alive until that work is enqueued.  The work
    goes on the stream that was current when it was handed over (autograd
    makes that the stream of the forward op); work from another stream
    flushes what is held first.  Every S_j ends bit-identical to the
    immediate path: the grouped launch, the
    shared-input call and the per-matrix call all give the same bits, and a
    second contribution to one S is added after the first, as in the
    backward's own order.  The inputs of a group are read once per weight
    here (once per group on the immediate path).  With `timing`, CUDA events
    bracket every flush on its stream (`events`, a list of (start, end)
    pairs)."""

    def __init__(self, flush_bytes: int = 8 << 30, timing: bool = False):
        self.flush_bytes = int(flush_bytes)
        self.timing = timing
        self.events = []
        self.flushes = 0
        self._pending = {}      # rank -> [targets]
        self._s_ptrs = set()
        self._bytes = 0
        self._ws = None
        self._plan = None
        self._stream = None
        self._ws_stream = None

    def __enter__(self):
        _active_batches.append(self)
        return self

    def __exit__(self, exc_type, exc, tb):
        _active_batches.remove(self)
        if exc_type is None:
            self.flush()
        else:
            self._pending.clear()
            self._s_ptrs.clear()
            self._bytes = 0
        return False

    def add(self, rank: int, targets) -> None:
        """targets: [(X, dY, S, seed, stream_id)] or [(X, dY, S, A)] of one rank."""
        stream = torch.cuda.current_stream(targets[0][0].device)
        if any(t[2].data_ptr() in self._s_ptrs for t in targets) or (self._stream is not None and
                                                                     stream != self._stream):
            self.flush()
        self._stream = stream
        self._pending.setdefault(rank, []).extend(targets)
        for t in targets:
            self._s_ptrs.add(t[2].data_ptr())
            self._bytes += t[0].numel() * t[0].element_size() + t[1].numel() * t[1].element_size()
        if self._bytes >= self.flush_bytes:
            self.flush()

    def _workspace(self, nbytes: int, device, stream) -> torch.Tensor:
        # the workspace and the plan's device buffer are reused only on the
        # stream whose earlier launches used them (stream order keeps the
        # reuse after those launches)
        if self._ws is not None and self._ws_stream != stream:
            self._ws = self._plan = None
        if self._ws is None or self._ws.numel() < nbytes or self._ws.device != device:
            self._ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
        self._ws_stream = stream
        return self._ws

    def flush(self) -> None:
        """Enqueues everything held, on the stream it arrived on."""
        for r, targets in self._pending.items():
            if not targets:
                continue
            device = targets[0][0].device
            st = self._stream
            with torch.cuda.stream(st):
                ws = self._workspace(logra_sketch_group_workspace_bytes(targets, r), device, st)
                plan = logra_sketch_group_plan(targets, r, workspace=ws, reuse=self._plan, stream=st)
                if self.timing:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                logra_sketch_accumulate_group(plan, stream=st)
                if self.timing:
                    e1.record(st)
                    self.events.append((e0, e1))
            self._plan = plan   # keeps the inputs alive until the next flush
            self.flushes += 1
        self._pending.clear()
        self._s_ptrs.clear()
        self._bytes = 0


class _SketchedLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, group, *weights):
        ctx.group = group
        ctx.save_for_backward(x, *weights)
        x2 = x.reshape(-1, x.shape[-1])
        return tuple((x2 @ w.t()).reshape(*x.shape[:-1], w.shape[0]) for w in weights)

    @staticmethod
    def backward(ctx, *grads):
        x, *weights = ctx.saved_tensors
        group = ctx.group
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        targets, grad_x = [], None
        for j, (g, w) in enumerate(zip(grads, weights)):
            if g is None:
                g = torch.zeros(*x.shape[:-1], w.shape[0], dtype=x.dtype, device=x.device)
            g2 = g.reshape(-1, w.shape[0]).contiguous().to(torch.bfloat16)
            if ctx.needs_input_grad[0]:
                gx = g2 @ w
                grad_x = gx if grad_x is None else grad_x + gx
            if group.operands is None:
                targets.append((g2, group.sketches[j], group.seeds[j], group.stream_ids[j]))
            else:
                targets.append((g2, group.sketches[j], group.operands[j]))
        if grad_x is not None:
            grad_x = grad_x.reshape(x.shape)
        batch = _current_batch()
        if batch is not None:
            # deferred: every weight a target of its own with the shared input
            batch.add(group.rank, [(x2,) + t for t in targets])
            return (grad_x, None) + (None,) * len(weights)
        # one call per run of weights whose stacked tiles fit (≤ 512 rows)
        per_call = max(1, 512 // ((group.rank + 15) // 16 * 16))
        ws = group._workspace(x2.shape[0], per_call)
        call = logra_sketch_accumulate_shared_x if group.operands is None else logra_sketch_accumulate_shared_x_proj
        for c in range(0, len(targets), per_call):
            call(x2, targets[c:c + per_call], group.rank, workspace=ws)
        return (grad_x, None) + (None,) * len(weights)


class SketchedLinearGroup(torch.nn.Module):
    """Bias-free bf16 linear maps y_j = x W_jᵀ that share their input x, with
    the weight gradients replaced by rank-r sketches.

    weights: list of (d_j × k) bf16 tensors (up to 4; when their stacked sign
             tiles exceed 512 rows the backward makes several calls)
    seeds, stream_ids: the projection A_j of each weight (regenerated, never stored)
    operands: optional list of bf16 (rank × k) projection operands Ã_j
             (A_j = Ã_j/√r), e.g. a Gaussian basis from logra_regen_projection;
             they replace the seeds when given
    """

    def __init__(self, weights, rank: int, seeds=None, stream_ids=None, operands=None):
        super().__init__()
        if not 1 <= len(weights) <= LOGRA_MAX_SHARED_X_TARGETS:
            raise ValueError("a group holds 1 to 4 weights")
        k = weights[0].shape[1]
        if any(w.shape[1] != k or w.dtype != torch.bfloat16 for w in weights):
            raise ValueError("the weights of a group are bf16 and share their input width")
        self.rank = rank
        if operands is None and (seeds is None or stream_ids is None):
            raise ValueError("give either seeds and stream_ids or operands")
        self.operands = list(operands) if operands is not None else None
        self.seeds = [int(s) for s in seeds] if seeds is not None else [0] * len(weights)
        self.stream_ids = [int(s) for s in stream_ids] if stream_ids is not None else [0] * len(weights)
        for j, w in enumerate(weights):
            self.register_buffer(f"weight{j}", w)
            self.register_buffer(f"sketch{j}", torch.zeros((w.shape[0], rank), dtype=torch.float32, device=w.device))
        self._ws = None

    @property
    def weights(self):
        return [getattr(self, f"weight{j}") for j in range(len(self.seeds))]

    @property
    def sketches(self):
        return [getattr(self, f"sketch{j}") for j in range(len(self.seeds))]

    def _workspace(self, T: int, per_call: int) -> torch.Tensor:
        w0 = self.weights[0]
        ds = [w.shape[0] for w in self.weights]
        need = max(1, max(logra_sketch_shared_x_workspace_bytes(T, w0.shape[1], ds[c:c + per_call], self.rank)
                          for c in range(0, len(ds), per_call)))
        if self._ws is None or self._ws.numel() < need or self._ws.device != w0.device:
            self._ws = torch.empty(need, dtype=torch.uint8, device=w0.device)
        return self._ws

    def forward(self, x: torch.Tensor):
        if x.dtype != torch.bfloat16:
            raise TypeError("input must be bfloat16")
        return _SketchedLinearFn.apply(x, self, *self.weights)

    @torch.no_grad()
    def merge_(self, alpha_eta, stream=None):
        """W_j ← bf16(W_j − αη·S_j·A_j) for every weight, then S_j = 0.
        alpha_eta: a float, or a device fp32 scalar tensor (e.g. from
        logra_step_size_device)."""
        dev_scalar = alpha_eta if isinstance(alpha_eta, torch.Tensor) else None
        ae = 0.0 if dev_scalar is not None else float(alpha_eta)
        # the merge and the clearing of its sketch run on one stream
        st = _torch_stream(stream, self.weights[0].device)
        with torch.cuda.stream(st):
            for j, (w, s, seed, sid) in enumerate(zip(self.weights, self.sketches, self.seeds, self.stream_ids)):
                if self.operands is None:
                    logra_merge_update(w, s, seed, sid, self.rank, ae, alpha_eta_dev=dev_scalar, stream=st)
                else:
                    logra_merge_update_proj(w, s, self.operands[j], self.rank, ae, alpha_eta_dev=dev_scalar,
                                            stream=st)
                s.zero_()


class GroupMerger:
    """Merges every weight of several `SketchedLinearGroup` modules (one common
    rank) in one launch, then clears their sketches.

    The plan (tensor maps and descriptors of every weight) is built on the
    first merge and kept while the groups' weight, sketch and operand buffers,
    seeds and stream ids stay the same; a change rebuilds it.  Groups with
    projection operands and groups with seeds go into separate plans (one
    launch each).  Each weight ends bit-identical to its group's `merge_`."""

    def __init__(self, groups):
        self.groups = list(groups)
        if not self.groups:
            raise ValueError("no groups to merge")
        self.rank = self.groups[0].rank
        if any(g.rank != self.rank for g in self.groups):
            raise ValueError("the groups of one merger share their rank")
        self._plans, self._key = [], None

    def _targets(self):
        seeded, given = [], []
        for g in self.groups:
            for j, (w, s) in enumerate(zip(g.weights, g.sketches)):
                if g.operands is None:
                    seeded.append((w, s, g.seeds[j], g.stream_ids[j]))
                else:
                    given.append((w, s, g.operands[j]))
        return [t for t in (seeded, given) if t]

    def _fingerprint(self, target_sets):
        return tuple(tuple((t[0].data_ptr(), t[1].data_ptr(), t[0].shape, t[1].stride(0))
                           + ((t[2], t[3]) if len(t) == 4 else (t[2].data_ptr(),)) for t in ts)
                     for ts in target_sets)

    @torch.no_grad()
    def merge_(self, alpha_eta, stream=None):
        """W ← bf16(W − αη·S·A) for every weight of every group, then S = 0.
        alpha_eta: a float, or a device fp32 scalar tensor."""
        target_sets = self._targets()
        # One torch stream for the plan copies, the merges and the clearing of
        # the sketches (a raw handle is wrapped), so the sketches are zeroed
        # only after the merges that read them.
        st = _torch_stream(stream, self.groups[0].weights[0].device)
        key = self._fingerprint(target_sets)
        if key != self._key:
            self._plans = [logra_merge_group_plan(ts, self.rank, stream=st) for ts in target_sets]
            self._key = key
        dev_scalar = alpha_eta if isinstance(alpha_eta, torch.Tensor) else None
        ae = 0.0 if dev_scalar is not None else float(alpha_eta)
        for plan in self._plans:
            logra_merge_update_group(plan, ae, alpha_eta_dev=dev_scalar, stream=st)
        sketches = [s for g in self.groups for s in g.sketches]
        with torch.cuda.stream(st):
            torch._foreach_zero_(sketches)
