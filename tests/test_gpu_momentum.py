"""Momentum on the sketch (M ← β·M + S) against the oracle, alone and ahead of
the merge (U = M)."""

import numpy as np
import pytest
import torch

import synthetic
from oracle import merge as omerge
from merge_tolerance import check as merge_check
from oracle import momentum as omom
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


def _check(got, ref):
    # one fused multiply-add rounded once to fp32: within half an fp32 ulp of
    # the exact value, which the fp64 oracle holds to 2^-53
    bound = 2.0**-24 * np.abs(ref) + 1e-45
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} elements outside one fp32 rounding"


@pytest.mark.parametrize("d,r", [(1000, 4), (333, 64), (129, 256), (1, 9)])
@pytest.mark.parametrize("beta", [0.0, 0.9, -0.5])
@pytest.mark.parametrize("clear_s", [False, True])
def test_momentum_matches_oracle(lg, d, r, beta, clear_s):
    g = torch.Generator(device=DEV).manual_seed(d * 7 + r)
    M = torch.randn((d, r), generator=g, device=DEV)
    S = torch.randn((d, r), generator=g, device=DEV) * 1e-2
    M0, S0 = _np(M), _np(S)
    lg.logra_sketch_momentum(M, S, beta, clear_s=clear_s)
    torch.cuda.synchronize()
    _check(_np(M), omom.momentum_update(M0, S0, float(np.float32(beta))))
    if clear_s:
        assert torch.count_nonzero(S) == 0
    else:
        assert np.array_equal(_np(S), S0)


def test_momentum_strided_rows(lg):
    # row strides above r take the row-walking kernel; bytes past column r stay
    g = torch.Generator(device=DEV).manual_seed(5)
    Mb = torch.randn((300, 72), generator=g, device=DEV)
    Sb = torch.randn((300, 70), generator=g, device=DEV)
    M, S = Mb[:, :64], Sb[:, :64]
    Mb0, Sb0 = Mb.clone(), Sb.clone()
    lg.logra_sketch_momentum(M, S, 0.95, clear_s=True)
    torch.cuda.synchronize()
    _check(_np(M), omom.momentum_update(_np(Mb0[:, :64]), _np(Sb0[:, :64]), float(np.float32(0.95))))
    assert torch.equal(Mb[:, 64:], Mb0[:, 64:]) and torch.equal(Sb[:, 64:], Sb0[:, 64:])
    assert torch.count_nonzero(S) == 0


def test_momentum_then_merge_over_three_steps(lg):
    # three steps of (sketch, momentum, merge) with a fixed projection; the
    # weight after each merge matches the oracle's merge with U = M_t
    d, k, r, beta, ae = 512, 1536, 64, 0.9, 5e-3
    seed, sid = 105, 2
    g = torch.Generator(device=DEV).manual_seed(1)
    W = (torch.randn((d, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    M = torch.zeros((d, r), device=DEV)
    A = oph.projection(seed, sid, r, k)
    Ss, W_ref = [], _np(W)
    for t in range(3):
        S = torch.randn((d, r), generator=g, device=DEV) * 0.05
        Ss.append(_np(S))
        M_prev = _np(M)
        lg.logra_sketch_momentum(M, S, beta, clear_s=True)
        lg.logra_merge_update(W, M, seed, sid, r, ae)
        torch.cuda.synchronize()
        # each step is one rounding of the oracle's update of the state the GPU holds
        _check(_np(M), omom.momentum_update(M_prev, Ss[-1], float(np.float32(beta))))
        # and the run stays within a few fp32 roundings per step of the exact recurrence
        M_run = omom.momentum_run(Ss, float(np.float32(beta)))
        assert np.abs(_np(M) - M_run).max() <= 4 * (t + 1) * 2.0**-24 * np.abs(M_run).max()
        ref = omerge.merge(W_ref, _np(M), A, float(np.float32(ae)))
        got = _np(W)
        merge_check(got, ref, W_ref, _np(M), A, float(np.float32(ae)))
        W_ref = got  # the next step starts from the bf16 weight the GPU holds


def test_momentum_full_sketch_buffer(lg):
    # the flat buffer holding every sketch of the 7B projection set at r = 64
    # (Σd = 1,390,592 rows): one launch, sampled rows checked
    w = synthetic.WORKLOADS["qwen7b"]
    rows = sum(d for (_, d, _, _) in w["layers"][0]) * len(w["layers"])
    r = 64
    g = torch.Generator(device=DEV).manual_seed(64)
    M = torch.randn((rows, r), generator=g, device=DEV)
    S = torch.randn((rows, r), generator=g, device=DEV) * 1e-3
    pick = np.unique(np.concatenate([[0, rows - 1], np.random.default_rng(3).integers(0, rows, 200)]))
    idx = torch.as_tensor(pick, device=DEV)
    M0, S0 = _np(M[idx]), _np(S[idx])
    lg.logra_sketch_momentum(M, S, 0.9, clear_s=True)
    torch.cuda.synchronize()
    _check(_np(M[idx]), omom.momentum_update(M0, S0, float(np.float32(0.9))))
    assert torch.count_nonzero(S) == 0
