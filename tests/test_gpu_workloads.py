"""Parity at the workloads' full sizes, in the launch configuration the bench
times (same entry points, same split plans, same kernels).

Sketches are checked on sampled rows (the oracle forms those rows of the
dense gradient explicitly); merges are checked on every weight; the predicted
KL is checked on sampled rows plus the identity q(D) = mean of the per-row KL
over all 65536 rows, and the controller's α is checked along the δ schedule.
"""

import math

import numpy as np
import pytest
import torch

import synthetic
from oracle import kl as okl
from oracle import merge as omerge
from merge_tolerance import check as merge_check
from oracle import philox as oph
from oracle import sketch as osk
from oracle import step as ostep

pytestmark = pytest.mark.gpu

DEV = "cuda"
S_TOL = 1e-3
Q_TOL = 1e-4


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


def _matrix(workload, name):
    for (n, d, k, sid) in synthetic.WORKLOADS[workload]["layers"][0]:
        if n == name:
            return d, k, sid
    raise KeyError(name)


def _sketch_rows_check(lg, workload, layer, name, r, nmb, nrows=12):
    w = synthetic.WORKLOADS[workload]
    d, k, sid = _matrix(workload, name)
    seed, T = w["seeds"][layer], w["tokens"]
    S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
    ws = lg.sketch_workspace(T, d, k, r, DEV)
    rng = np.random.default_rng(layer * 31 + r)
    rows = np.unique(np.concatenate([[0, d - 1], rng.integers(0, d, nrows)]))
    mbs = []
    for m in range(nmb):
        X, dY = synthetic.microbatch(workload, layer, name, m, T, d, k, DEV)
        lg.logra_sketch_accumulate(X, dY, S, seed, sid, r, ws)
        mbs.append((_np(X), _np(dY[:, rows])))
        del X, dY
    torch.cuda.synchronize()
    A = oph.projection(seed, sid, r, k)
    ref = osk.sketch_rows(np.zeros((len(rows), r)), np.arange(len(rows)), mbs, A)
    rel = _rel(_np(S)[rows], ref)
    assert rel <= S_TOL, rel
    assert torch.isfinite(S).all()
    return S


def _merge_full_check(lg, workload, layer, name, r, S):
    w = synthetic.WORKLOADS[workload]
    d, k, sid = _matrix(workload, name)
    seed, ae = w["seeds"][layer], w["alpha_eta"]
    W = synthetic.weight(workload, layer, name, d, k, DEV)
    W0 = _np(W)
    lg.logra_merge_update(W, S, seed, sid, r, ae)
    torch.cuda.synchronize()
    S_np = _np(S)
    A = oph.projection(seed, sid, r, k)
    ae32 = float(np.float32(ae))
    ref = omerge.merge(W0, S_np, A, ae32)
    got = _np(W)
    # every weight within the bound; the ones outside a strict 1-ulp bound
    # (printed; about one in a million here) are all cancellations
    n_allow = merge_check(got, ref, W0, S_np, A, ae32, what=f"{workload} {name} r={r}")
    print(f"[merge tolerance] {workload} {name} {d}x{k} r={r}: {n_allow} of {got.size} weights outside a strict "
          "1-ulp bound, all cancellations")
    assert n_allow <= 4 + 2 * got.size // 10**6
    assert np.mean(got != W0) > 1e-3  # the update is visible in bf16


# 1.5B-class set: the rank sweep r ∈ {4, 16, 64, 256}, 4 micro-batches of
# 8192 tokens, per-layer seed 100 + layer; each rank on a different matrix so
# that every shape family and ranks below and above the MMA width of 16 run.
@pytest.mark.parametrize("name,r,layer", [("gate", 4, 3), ("down", 16, 11), ("q", 64, 17), ("k", 256, 27)])
def test_qwen15b_rank_sweep(lg, name, r, layer):
    S = _sketch_rows_check(lg, "qwen1.5b", layer, name, r, nmb=4)
    _merge_full_check(lg, "qwen1.5b", layer, name, r, S)


# 7B-class set: r ∈ {256, 64}; eight micro-batches of 16384 tokens on a value
# projection, then the merge.
@pytest.mark.parametrize("r", [64, 256])
def test_qwen7b_eight_microbatches(lg, r):
    S = _sketch_rows_check(lg, "qwen7b", 13, "v", r, nmb=8)
    _merge_full_check(lg, "qwen7b", 13, "v", r, S)


@pytest.mark.parametrize("r", [64, 256])
def test_qwen7b_gate_merge_full(lg, r):
    # the largest weight of the set (18944 × 3584), every element checked
    d, k, _ = _matrix("qwen7b", "gate")
    S = torch.randn((d, r), generator=torch.Generator(device=DEV).manual_seed(r), device=DEV) * 0.05
    _merge_full_check(lg, "qwen7b", 0, "gate", r, S)


@pytest.mark.parametrize("eps", [0.01, 0.1])
def test_predicted_kl_full_workload(lg, eps):
    kw = synthetic.KL_WORKLOADS["qwen"]
    cur, prop = synthetic.kl_logits("qwen", eps, device=DEV)  # 65536 × 151936 bf16
    rows = cur.shape[0]
    row_kl = torch.empty(rows, dtype=torch.float32, device=DEV)
    q_dev = lg.logra_predicted_kl(cur, prop, kw["temperature"], row_kl_out=row_kl)
    torch.cuda.synchronize()
    q = float(q_dev.item())
    rk = row_kl.double().cpu().numpy()
    # q(D) is the mean of the per-row values (row values are rounded to fp32 on output)
    assert abs(q - rk.mean()) <= 1e-6 * q
    assert np.all(rk >= 0)
    rng = np.random.default_rng(int(eps * 1000))
    sample = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, 30)]))
    _, ref = okl.predicted_kl(_np(cur[sample]), _np(prop[sample]), kw["temperature"])
    assert np.allclose(rk[sample], ref, rtol=Q_TOL, atol=0)
    # the controller along the annealed budget, on the host and on the device
    ae = torch.empty((), dtype=torch.float32, device=DEV)
    al = torch.empty((), dtype=torch.float64, device=DEV)
    for delta in lg.delta_schedule(kw["delta"][0], kw["delta"][1], kw["steps"]):
        want = ostep.step_size(q, delta, kw["alpha_max"])
        assert lg.logra_step_size(q, delta, kw["alpha_max"]) == want
        lg.logra_step_size_device(q_dev, delta, kw["alpha_max"], 1.0, ae, al)
        assert float(al.item()) == want
