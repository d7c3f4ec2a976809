"""Refreshed and Gaussian projections against the oracle: the Gaussian operand
from the regen kernel, sketches and merges with a given projection operand,
and per-step seeds."""

import numpy as np
import pytest
import torch

import synthetic
from oracle import gaussian as og
from oracle import merge as omerge
from merge_tolerance import check as merge_check
from oracle import philox as oph
from oracle import sketch as osk

pytestmark = pytest.mark.gpu
DEV = "cuda"
S_TOL = 1e-3


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


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _check_operand(got, seed, sid, r, k):
    """got (fp64 values of the GPU's bf16 operand) against bf16_rn(z) of the oracle.

    The GPU evaluates z in fp32, so where the exact z lies within a few fp32
    ulps of a bf16 rounding midpoint either neighbour is correct; everywhere
    else the two roundings must agree exactly."""
    z = og.normals(seed, sid, r, k)
    ref = omerge.bf16_round(z)
    diff = got != ref
    if diff.any():
        # the two bf16 neighbours of z around the midpoint between them
        ulp = omerge.bf16_ulp(ref)
        lo, hi = np.minimum(got, ref), np.maximum(got, ref)
        mid = (lo + hi) / 2
        near = np.abs(z - mid) <= 2.0**-20 * np.abs(z)
        adjacent = np.abs(hi - lo) <= ulp * 1.0000001
        assert np.all(near[diff] & adjacent[diff]), "operand differs away from a rounding midpoint"
    assert diff.mean() < 1e-3
    return ref


@pytest.mark.parametrize("r,k", [(1, 5), (9, 1001), (64, 3584), (256, 1536)])
def test_gaussian_operand_matches_oracle(lg, r, k):
    seed, sid = 2024 + r, 3
    A = lg.logra_regen_projection(seed, sid, r, k, lg.LOGRA_PROJ_GAUSS_BF16)
    A32 = lg.logra_regen_projection(seed, sid, r, k, lg.LOGRA_PROJ_GAUSS_FP32)
    torch.cuda.synchronize()
    got = _np(A)
    _check_operand(got, seed, sid, r, k)
    # the fp32 kind is the same operand scaled by 1/√r (one rounding)
    assert np.allclose(_np(A32), got / np.sqrt(r), rtol=2.0**-23, atol=0)


def _gauss_operand(lg, seed, sid, r, k):
    A = lg.logra_regen_projection(seed, sid, r, k, lg.LOGRA_PROJ_GAUSS_BF16)
    torch.cuda.synchronize()
    return A, _check_operand(_np(A), seed, sid, r, k)


@pytest.mark.parametrize("T,d,k,r", [(1000, 136, 200, 9), (384, 512, 1536, 64), (700, 264, 520, 256), (129, 64, 64, 4)])
def test_sketch_with_gaussian_operand(lg, T, d, k, r):
    seed, sid = 77, 5
    A, A_ref = _gauss_operand(lg, seed, sid, r, k)
    X, dY = synthetic.microbatch("tiny", 0, "g", 0, T, d, k, DEV)
    S = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate_proj(X, dY, S, A, r)
    lg.logra_sketch_accumulate_proj(X, dY, S, A, r)  # accumulates
    torch.cuda.synchronize()
    ref = osk.sketch_accumulate(np.zeros((d, r)), [(_np(X), _np(dY))] * 2, A_ref / np.sqrt(r))
    assert _rel(_np(S), ref) <= S_TOL
    assert torch.isfinite(S).all()


@pytest.mark.parametrize("T,d,k,r", [(1000, 256, 1536, 64), (300, 136, 520, 256), (256, 64, 128, 16)])
def test_sketch_with_sign_operand_equals_generated_signs(lg, T, d, k, r):
    # the ±1 signs passed as an operand take the TMA path for the B tiles and
    # must reproduce the on-chip generated tiles bit for bit
    seed, sid = 105, 2
    signs = torch.as_tensor(oph.signs(seed, sid, r, k), device=DEV).to(torch.bfloat16).contiguous()
    X, dY = synthetic.microbatch("tiny", 0, "s", 0, T, d, k, DEV)
    S1 = torch.zeros((d, r), device=DEV)
    S2 = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate(X, dY, S1, seed, sid, r)
    lg.logra_sketch_accumulate_proj(X, dY, S2, signs, r)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2)


@pytest.mark.parametrize("d,k,r", [(300, 520, 4), (129, 1000, 8), (256, 1536, 64), (200, 264, 256), (1, 8, 16)])
def test_merge_with_gaussian_operand(lg, d, k, r):
    seed, sid, ae = 31, 1, 3e-3
    A, A_ref = _gauss_operand(lg, seed, sid, r, k)
    g = torch.Generator(device=DEV).manual_seed(d + r)
    W = (torch.randn((d, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    S = torch.randn((d, r), generator=g, device=DEV) * 0.05
    W0 = _np(W)
    lg.logra_merge_update_proj(W, S, A, r, ae)
    torch.cuda.synchronize()
    ae32 = float(np.float32(ae))
    ref = omerge.merge(W0, _np(S), A_ref / np.sqrt(r), ae32)
    merge_check(_np(W), ref, W0, _np(S), A_ref / np.sqrt(r), ae32)


@pytest.mark.parametrize("d,k,r", [(256, 1536, 64), (200, 520, 256), (129, 1000, 8)])
def test_merge_with_sign_operand(lg, d, k, r):
    seed, sid, ae = 105, 4, 2e-2
    signs = torch.as_tensor(oph.signs(seed, sid, r, k), device=DEV).to(torch.bfloat16).contiguous()
    g = torch.Generator(device=DEV).manual_seed(d * r)
    W = (torch.randn((d, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    S = torch.randn((d, r), generator=g, device=DEV) * 0.05
    W1, W2 = W.clone(), W.clone()
    lg.logra_merge_update(W1, S, seed, sid, r, ae)
    lg.logra_merge_update_proj(W2, S, signs, r, ae)
    torch.cuda.synchronize()
    assert torch.equal(W1, W2)  # same tensor-core sequence, tiles from TMA instead of the generator
    ae32 = float(np.float32(ae))
    A_ref = oph.projection(seed, sid, r, k)
    ref = omerge.merge(_np(W), _np(S), A_ref, ae32)
    merge_check(_np(W2), ref, _np(W), _np(S), A_ref, ae32)


def test_refreshed_basis_steps(lg):
    # step t sketches with seed_t = refreshed(base, t): each step matches the
    # oracle with that step's projection, and consecutive steps differ
    base, sid, T, d, k, r = 105, 0, 512, 256, 1536, 16
    X, dY = synthetic.microbatch("tiny", 0, "rf", 0, T, d, k, DEV)
    out = []
    for t in range(3):
        seed_t = lg.logra_refreshed_seed(base, t)
        S = torch.zeros((d, r), device=DEV)
        lg.logra_sketch_accumulate(X, dY, S, seed_t, sid, r)
        torch.cuda.synchronize()
        ref = osk.sketch_accumulate(np.zeros((d, r)), [(_np(X), _np(dY))],
                                    oph.projection(oph.refreshed_seed(base, t), sid, r, k))
        assert _rel(_np(S), ref) <= S_TOL
        out.append(_np(S))
    assert _rel(out[0], out[1]) > 0.5


def test_gaussian_full_size_down_projection(lg):
    # 7B down projection (d = 3584, k = 18944) at r = 256 with a Gaussian
    # basis: operand of 4.6 MiB, one 16384-token micro-batch, sampled rows
    w = synthetic.WORKLOADS["qwen7b"]
    name, d, k, sid = [m for m in w["layers"][0] if m[0] == "down"][0]
    r, seed, T = 256, w["seeds"][5], w["tokens"]
    A, A_ref = _gauss_operand(lg, seed, sid, r, k)
    X, dY = synthetic.microbatch("qwen7b", 5, name, 0, T, d, k, DEV)
    S = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate_proj(X, dY, S, A, r)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, d - 1], np.random.default_rng(5).integers(0, d, 10)]))
    ref = osk.sketch_rows(np.zeros((len(rows), r)), np.arange(len(rows)), [(_np(X), _np(dY[:, rows]))],
                          A_ref / np.sqrt(r))
    assert _rel(_np(S)[rows], ref) <= S_TOL
