"""The sketch of a set of matrices with one launch per phase
(logra_sketch_accumulate_group), through the C ABI: every target's S equals
the per-matrix call bit for bit, and the fp64 oracle within the sketch bound.

LoGRA summary page, section "草图如何取代完整梯度缓冲": each sketched weight
adds its micro-batch contribution into its own S during the backward pass.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import philox as oph
from oracle import sketch as osk

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def lg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_gradient_sketching_gb300 as mod

    torch.cuda.set_device(0)
    assert mod.logra_device_error() == 0
    yield mod
    assert mod.logra_device_error() == 0


def _np(t):
    return t.detach().double().cpu().numpy()


def _pad(t, mult=8):
    rows, cols = t.shape
    ld = (cols + mult - 1) // mult * mult
    if ld == cols:
        return t
    buf = torch.zeros((rows, ld), dtype=t.dtype, device=t.device)
    buf[:, :cols] = t
    return buf[:, :cols]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _tight(r):
    return 1e-4 if r <= 64 else 4e-4


# (T, d, k): ragged tails on every tile size, less than one tile, many split
# ranges of T (4096 × 256), a wide k, one token, and empty targets.
SHAPES = [(1000, 304, 520), (128, 256, 256), (77, 64, 64), (4096, 256, 512), (0, 64, 64), (300, 136, 200),
          (1, 8, 8), (640, 1000, 200), (128, 0, 64), (512, 384, 640)]


def _targets(shapes, r, tag, operands=False):
    """[(X, dY, S, seed, sid)] or [(X, dY, S, A)] with seeded inputs and a
    seeded nonzero start for S (every S its own buffer)."""
    out = []
    for j, (T, d, k) in enumerate(shapes):
        X, dY = synthetic.microbatch("tiny", 0, f"{tag}{j}", 0, T, d, k, DEV)
        X, dY = _pad(X), _pad(dY)
        S = torch.randn((d, r), generator=torch.Generator(device=DEV).manual_seed(40 + j), device=DEV) * 1e-3
        if operands:
            A = torch.randn((r, k), generator=torch.Generator(device=DEV).manual_seed(70 + j), device=DEV)
            out.append((X, dY, S, A.to(torch.bfloat16)))
        else:
            out.append((X, dY, S, 1000 + 17 * j, j % 7))
    return out


def _per_matrix(lg, targets, r):
    """Every target's S after one per-matrix call (copies; the inputs stay)."""
    res = []
    for t in targets:
        X, dY, S = t[0], t[1], t[2].clone()
        T, k = X.shape
        ws = lg.sketch_workspace(T, dY.shape[1], k, r, DEV)
        if len(t) == 5:
            lg.logra_sketch_accumulate(X, dY, S, t[3], t[4], r, ws)
        else:
            lg.logra_sketch_accumulate_proj(X, dY, S, t[3], r, ws)
        res.append(S)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("r", [1, 4, 16, 64, 100, 256])
def test_group_equals_per_matrix_calls(lg, r):
    targets = _targets(SHAPES, r, f"g{r}-")
    want = _per_matrix(lg, targets, r)
    plan = lg.logra_sketch_group_plan(targets, r)
    lg.logra_sketch_accumulate_group(plan)
    torch.cuda.synchronize()
    for j, (t, w) in enumerate(zip(targets, want)):
        assert torch.equal(t[2], w), (j, SHAPES[j])


@pytest.mark.parametrize("r", [16, 64, 256])
def test_group_matches_oracle(lg, r):
    shapes = [(1000, 304, 520), (300, 136, 200), (77, 64, 64), (4096, 256, 512)]
    targets = _targets(shapes, r, f"o{r}-")
    S0 = [_np(t[2]) for t in targets]
    plan = lg.logra_sketch_group_plan(targets, r)
    lg.logra_sketch_accumulate_group(plan)
    torch.cuda.synchronize()
    for (X, dY, S, seed, sid), s0 in zip(targets, S0):
        ref = osk.sketch_accumulate(s0, [(_np(X), _np(dY))], oph.projection(seed, sid, r, X.shape[1]))
        rel = _rel(_np(S), ref)
        assert rel <= _tight(r), rel


@pytest.mark.parametrize("r", [16, 256])
def test_group_with_given_operands(lg, r):
    # targets with a given projection operand and targets with signs from the
    # seed in one plan: each equals its own per-matrix call
    a = _targets(SHAPES[:5], r, f"a{r}-", operands=True)
    b = _targets(SHAPES[5:], r, f"b{r}-")
    targets = [t for pair in zip(a, b) for t in pair]
    want = _per_matrix(lg, targets, r)
    plan = lg.logra_sketch_group_plan(targets, r)
    lg.logra_sketch_accumulate_group(plan)
    torch.cuda.synchronize()
    for j, (t, w) in enumerate(zip(targets, want)):
        assert torch.equal(t[2], w), j


def test_group_plan_reuse_accumulates(lg):
    # the plan stays valid while its buffers do: two launches add two
    # contributions, as two per-matrix calls do
    r = 64
    targets = _targets(SHAPES[:4], r, "re-")
    want = [w.clone() for w in _per_matrix(lg, targets, r)]
    for t, w in zip(targets, want):
        ws = lg.sketch_workspace(t[0].shape[0], t[1].shape[1], t[0].shape[1], r, DEV)
        lg.logra_sketch_accumulate(t[0], t[1], w, t[3], t[4], r, ws)
    plan = lg.logra_sketch_group_plan(targets, r)
    lg.logra_sketch_accumulate_group(plan)
    lg.logra_sketch_accumulate_group(plan)
    torch.cuda.synchronize()
    for t, w in zip(targets, want):
        assert torch.equal(t[2], w)


def test_group_of_nothing(lg):
    r = 16
    targets = _targets([(0, 64, 64), (128, 0, 64), (64, 64, 0)], r, "e-")
    before = [t[2].clone() for t in targets]
    plan = lg.logra_sketch_group_plan(targets, r)
    assert plan.workspace.numel() == 1
    lg.logra_sketch_accumulate_group(plan)
    lg.logra_sketch_accumulate_group(lg.logra_sketch_group_plan([], r, device=DEV))
    torch.cuda.synchronize()
    for t, b in zip(targets, before):
        assert torch.equal(t[2], b)


def test_group_refuses_a_sketch_named_twice(lg):
    r = 16
    targets = _targets(SHAPES[:2], r, "dup-")
    targets[1] = (targets[1][0], targets[1][1], targets[0][2][: targets[1][1].shape[1]], 5, 1)
    with pytest.raises(lg.LograError, match="overlap"):
        lg.logra_sketch_group_plan(targets, r)


@pytest.mark.parametrize("r", [64, 256])
def test_group_qwen7b_layer(lg, r):
    # the seven projections of one 7B decoder layer at the full micro-batch
    # (16384 tokens) in one plan, against one call per matrix
    w = synthetic.WORKLOADS["qwen7b"]
    layer, T = 3, w["tokens"]
    targets = []
    for (name, d, k, sid) in w["layers"][layer]:
        X, dY = synthetic.microbatch("qwen7b", layer, name, 0, T, d, k, DEV)
        S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
        targets.append((X, dY, S, w["seeds"][layer], sid))
    want = _per_matrix(lg, targets, r)
    plan = lg.logra_sketch_group_plan(targets, r)
    lg.logra_sketch_accumulate_group(plan)
    torch.cuda.synchronize()
    for (name, *_), t, ww in zip(w["layers"][layer], targets, want):
        assert torch.equal(t[2], ww), name
    # and one matrix against the oracle on sampled rows of S
    X, dY, S, seed, sid = targets[1]  # k: 512 × 3584
    rows = torch.arange(0, dY.shape[1], 37)
    A = oph.projection(seed, sid, r, X.shape[1])
    ref = osk.sketch_accumulate(np.zeros((len(rows), r)), [(_np(X), _np(dY[:, rows]))], A)
    assert _rel(_np(S[rows]), ref) <= _tight(r)


@pytest.mark.parametrize("r", [16, 100])
def test_group_of_many_small_matrices(lg, r):
    # more matrices than a CTA has threads (the launches find their matrix by
    # a binary search over the plan), with empty ones among them
    rng = np.random.default_rng(r)
    shapes = []
    for j in range(450):
        T = int(rng.choice([0, 8, 64, 200]))
        d = int(rng.choice([0, 8, 64, 136]))
        k = int(rng.choice([8, 64, 96]))
        shapes.append((T, d, k))
    targets = _targets(shapes, r, f"many{r}-")
    want = _per_matrix(lg, targets, r)
    plan = lg.logra_sketch_group_plan(targets, r)
    lg.logra_sketch_accumulate_group(plan)
    torch.cuda.synchronize()
    for j, (t, w) in enumerate(zip(targets, want)):
        assert torch.equal(t[2], w), (j, shapes[j])
