"""Merge of a set of weights in one launch: every weight equals its own
per-weight merge bit for bit (same arithmetic), and the oracle on a small
set."""

import numpy as np
import pytest
import torch

import synthetic
from oracle import merge as omerge
from merge_tolerance import check as merge_check
from oracle import philox as oph

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
    yield mod
    assert mod.logra_device_error() == 0


def _np(t):
    return t.detach().double().cpu().numpy()


# ragged rows and columns, a single row, an empty weight, several tiles
SHAPES = [(300, 520), (1, 8), (129, 1000), (0, 64), (256, 1536), (64, 0), (1000, 264)]


def _set(shapes, r, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    Ws, Ss = [], []
    for d, k in shapes:
        Ws.append((torch.randn((d, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16))
        Ss.append(torch.randn((d, r), generator=g, device=DEV) * 0.05)
    return Ws, Ss


@pytest.mark.parametrize("r", [4, 8, 16, 64, 100, 256])
def test_group_equals_per_weight_merges(lg, r):
    Ws, Ss = _set(SHAPES, r, r)
    ref = [W.clone() for W in Ws]
    ae = 3e-3
    for j, (W, S) in enumerate(zip(ref, Ss)):
        lg.logra_merge_update(W, S, 1000 + j, j, r, ae)
    plan = lg.logra_merge_group_plan([(W, S, 1000 + j, j) for j, (W, S) in enumerate(zip(Ws, Ss))], r)
    lg.logra_merge_update_group(plan, ae)
    torch.cuda.synchronize()
    for W, R in zip(Ws, ref):
        assert torch.equal(W, R)


@pytest.mark.parametrize("r", [8, 64, 256])
def test_group_with_operands_equals_per_weight(lg, r):
    shapes = [(300, 520), (129, 1000), (256, 1536)]
    Ws, Ss = _set(shapes, r, 7 * r)
    ops = [lg.logra_regen_projection(50 + j, j, r, k, lg.LOGRA_PROJ_GAUSS_BF16) for j, (_, k) in enumerate(shapes)]
    ref = [W.clone() for W in Ws]
    for W, S, A in zip(ref, Ss, ops):
        lg.logra_merge_update_proj(W, S, A, r, 2e-3)
    plan = lg.logra_merge_group_plan(list(zip(Ws, Ss, ops)), r)
    lg.logra_merge_update_group(plan, 2e-3)
    torch.cuda.synchronize()
    for W, R in zip(Ws, ref):
        assert torch.equal(W, R)


@pytest.mark.parametrize("r", [4, 64])
def test_group_plan_reuse_and_device_step(lg, r):
    # one plan, two steps: αη from the host, then from device memory; S is
    # rewritten in place between the steps (the plan holds pointers)
    Ws, Ss = _set(SHAPES[:3], r, 11)
    ref = [W.clone() for W in Ws]
    plan = lg.logra_merge_group_plan([(W, S, 5, j) for j, (W, S) in enumerate(zip(Ws, Ss))], r)
    ae_dev = torch.tensor([4e-3], device=DEV)
    for step in range(2):
        for j, (W, S) in enumerate(zip(ref, Ss)):
            lg.logra_merge_update(W, S, 5, j, r, 1e-3, alpha_eta_dev=ae_dev if step else None)
        lg.logra_merge_update_group(plan, 1e-3, alpha_eta_dev=ae_dev if step else None)
        for S in Ss:
            S.mul_(-0.5)
    torch.cuda.synchronize()
    for W, R in zip(Ws, ref):
        assert torch.equal(W, R)


@pytest.mark.parametrize("r", [4, 16])
def test_group_matches_oracle(lg, r):
    shapes = [(300, 520), (129, 264)]
    Ws, Ss = _set(shapes, r, 3)
    W0 = [_np(W) for W in Ws]
    ae = 5e-3
    plan = lg.logra_merge_group_plan([(W, S, 77, 10 + j) for j, (W, S) in enumerate(zip(Ws, Ss))], r)
    lg.logra_merge_update_group(plan, ae)
    torch.cuda.synchronize()
    ae32 = float(np.float32(ae))
    for j, (W, S) in enumerate(zip(Ws, Ss)):
        k = W.shape[1]
        A = oph.projection(77, 10 + j, r, k)
        ref = omerge.merge(W0[j], _np(S), A, ae32)
        merge_check(_np(W), ref, W0[j], _np(S), A, ae32)


@pytest.mark.parametrize("r", [4, 64, 256])
def test_group_full_15b_set(lg, r):
    # all 196 weights of the 1.5B projection set in one launch against the
    # per-weight merges (seeds and stream ids of the set)
    w = synthetic.WORKLOADS["qwen1.5b"]
    mats = [(layer, name, d, k, sid) for layer, ms in enumerate(w["layers"]) for (name, d, k, sid) in ms]
    g = torch.Generator(device=DEV).manual_seed(r)
    Ws = [(torch.randn((d, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16) for (_, _, d, k, _) in mats]
    Ss = [torch.randn((d, r), generator=g, device=DEV) * 1e-3 for (_, _, d, _, _) in mats]
    ref = [W.clone() for W in Ws]
    for (layer, _, _, _, sid), W, S in zip(mats, ref, Ss):
        lg.logra_merge_update(W, S, w["seeds"][layer], sid, r, 2e-4)
    plan = lg.logra_merge_group_plan([(W, S, w["seeds"][layer], sid)
                                      for (layer, _, _, _, sid), W, S in zip(mats, Ws, Ss)], r)
    lg.logra_merge_update_group(plan, 2e-4)
    torch.cuda.synchronize()
    assert all(torch.equal(W, R) for W, R in zip(Ws, ref))


@pytest.mark.parametrize("r", [64, 256])
def test_group_plan_rewritten_in_place(lg, r):
    # a second plan copied into the device buffer of the first: the kernels
    # must read the new tensor maps, not descriptors of the earlier plan (whose
    # weights stay alive here, so a stale map would only show as a mismatch)
    shapes = [(300, 520), (256, 1536), (129, 1000)]
    Wa, Sa = _set(shapes, r, 21)
    Wb, Sb = _set(shapes[::-1], r, 22)
    refa, refb = [W.clone() for W in Wa], [W.clone() for W in Wb]
    for j, (W, S) in enumerate(zip(refa, Sa)):
        lg.logra_merge_update(W, S, 3, j, r, 1e-3)
    for j, (W, S) in enumerate(zip(refb, Sb)):
        lg.logra_merge_update(W, S, 4, j, r, 1e-3)
    pa = lg.logra_merge_group_plan([(W, S, 3, j) for j, (W, S) in enumerate(zip(Wa, Sa))], r)
    lg.logra_merge_update_group(pa, 1e-3)
    pb = lg.logra_merge_group_plan([(W, S, 4, j) for j, (W, S) in enumerate(zip(Wb, Sb))], r, reuse=pa)
    assert pb.dev.data_ptr() == pa.dev.data_ptr()
    lg.logra_merge_update_group(pb, 1e-3)
    torch.cuda.synchronize()
    assert all(torch.equal(W, R) for W, R in zip(Wa, refa))
    assert all(torch.equal(W, R) for W, R in zip(Wb, refb))


@pytest.mark.parametrize("r", [4, 64, 256])
def test_group_plan_layout(lg, r):
    # the host copy of a plan: header, per-weight first CTA, and the split of
    # each weight into 128-row tiles × column ranges of at most 32 chunks
    import struct

    Ws, Ss = _set(SHAPES, r, 5)
    plan = lg.logra_merge_group_plan([(W, S, 1, j) for j, (W, S) in enumerate(zip(Ws, Ss))], r)
    raw = plan.host.cpu().numpy().tobytes()
    magic, n, r_, np_, path, total = struct.unpack_from("<Iiiiii", raw, 0)
    np_expect = (r + 15) // 16 * 16
    assert (magic, n, r_, np_, path) == (0x4C474D50, len(SHAPES), r, np_expect, 1 if np_expect <= 128 else 2)
    ctas = []
    for d, k in SHAPES:
        if d == 0 or k == 0:
            ctas.append(0)
            continue
        nc = (k + 63) // 64
        g = (nc + 31) // 32
        cpc = max((nc + g - 1) // g, min(nc, max(1, np_expect // 16)))
        ctas.append((d + 127) // 128 * ((nc + cpc - 1) // cpc))
    begin = struct.unpack_from(f"<{n + 1}i", raw, 128)
    assert list(begin) == [sum(ctas[:j]) for j in range(n + 1)] and total == sum(ctas)


@pytest.mark.parametrize("r", [8, 64, 200, 256])
@pytest.mark.parametrize("pad_s", [0, 1])
def test_group_strided_weights_and_sketches(lg, r, pad_s):
    # W as column slices of wider buffers (ldw > k) and S with row stride
    # r + pad_s: an odd stride keeps S out of the TMA staging path (above
    # r = 128 the first epilogue group then loads it while the second starts)
    shapes = [(300, 520), (129, 1000), (256, 64)]
    g = torch.Generator(device=DEV).manual_seed(r + pad_s)
    Wb = [(torch.randn((d, k + 24), generator=g, device=DEV) * 0.02).to(torch.bfloat16) for d, k in shapes]
    Sb = [torch.randn((d, r + pad_s), generator=g, device=DEV) * 0.05 for d, _ in shapes]
    Ws = [w[:, :k] for w, (_, k) in zip(Wb, shapes)]
    Ss = [s[:, :r] for s in Sb]
    refb = [w.clone() for w in Wb]
    for j, (R, S, (_, k)) in enumerate(zip(refb, Ss, shapes)):
        lg.logra_merge_update(R[:, :k], S, 8, j, r, 2e-3)
    plan = lg.logra_merge_group_plan([(W, S, 8, j) for j, (W, S) in enumerate(zip(Ws, Ss))], r)
    lg.logra_merge_update_group(plan, 2e-3)
    torch.cuda.synchronize()
    for W, R in zip(Wb, refb):
        assert torch.equal(W, R)  # the columns past k are untouched in both
    ae32 = float(np.float32(2e-3))
    W0 = (torch.randn((300, 520 + 24), generator=torch.Generator(device=DEV).manual_seed(r + pad_s), device=DEV)
          * 0.02).to(torch.bfloat16)[:, :520]
    A = oph.projection(8, 0, r, 520)
    ref = omerge.merge(_np(W0), _np(Ss[0]), A, ae32)
    merge_check(_np(Ws[0]), ref, _np(W0), _np(Ss[0]), A, ae32)


@pytest.mark.parametrize("r", [16, 256])
def test_group_of_many_small_weights(lg, r):
    # more weights than a CTA has threads (each CTA finds its weight by a
    # binary search over the plan), with empty ones among them
    rng = np.random.default_rng(r + 1)
    shapes = [(int(rng.choice([0, 8, 100, 300])), int(rng.choice([0, 8, 72, 136]))) for _ in range(500)]
    Ws, Ss = _set(shapes, r, r + 7)
    ref = [W.clone() for W in Ws]
    ae = 2e-3
    for j, (W, S) in enumerate(zip(ref, Ss)):
        lg.logra_merge_update(W, S, 50 + j, j % 7, r, ae)
    plan = lg.logra_merge_group_plan([(W, S, 50 + j, j % 7) for j, (W, S) in enumerate(zip(Ws, Ss))], r)
    lg.logra_merge_update_group(plan, ae)
    torch.cuda.synchronize()
    for j, (W, R) in enumerate(zip(Ws, ref)):
        assert torch.equal(W, R), (j, shapes[j])


@pytest.mark.parametrize("r", [64, 256])
@pytest.mark.parametrize("d,k", [(18944, 3584), (3584, 18944)])
def test_sign_operand_equals_on_chip_signs_full_size(lg, r, d, k):
    # The given-operand path with the sign operand of the same (seed, stream)
    # runs the same arithmetic as the on-chip signs, so the two agree bit for
    # bit.  At the 7B gate and down shapes a CTA runs 28-60 chunks with both
    # MMA issuers above r = 128, whose operand tiles arrive by TMA (out of
    # order when they like): repeated launches, one weight and in a plan.
    g = torch.Generator(device=DEV).manual_seed(r + d)
    W = (torch.randn((d, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    S = torch.randn((d, r), generator=g, device=DEV) * 0.05
    seed, sid, ae = 4242, 5, 3e-3
    A = lg.logra_regen_projection(seed, sid, r, k, lg.LOGRA_PROJ_SIGN_BF16)
    w_chip, w_op = W.clone(), W.clone()
    for _ in range(3):
        lg.logra_merge_update(w_chip, S, seed, sid, r, ae)
        lg.logra_merge_update_proj(w_op, S, A, r, ae)
    torch.cuda.synchronize()
    assert lg.logra_device_error() == 0
    assert torch.equal(w_chip, w_op)
    w_grp = W.clone()
    plan = lg.logra_merge_group_plan([(w_grp, S, A)], r)
    for _ in range(3):
        lg.logra_merge_update_group(plan, ae)
    torch.cuda.synchronize()
    assert lg.logra_device_error() == 0
    assert torch.equal(w_grp, w_chip)
