"""Gradient-reconstruction diagnostic and the sum-of-squares kernel against
the oracle."""

import numpy as np
import pytest
import torch

import synthetic
from oracle import diagnostic as odiag
from oracle import gaussian as og
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


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,cols,ld", [(1, 1, 1), (1000, 37, 40), (3, 70000, 70000), (0, 5, 5), (18944, 512, 512)])
def test_sum_squares_matches_fp64(lg, dtype, rows, cols, ld):
    g = torch.Generator(device=DEV).manual_seed(rows + cols)
    buf = (torch.randn((max(rows, 1), ld), generator=g, device=DEV) * 3).to(dtype)
    x = buf[:rows, :cols]
    out = torch.full((1,), 5.0, dtype=torch.float64, device=DEV)
    lg.logra_sum_squares(x, out)
    torch.cuda.synchronize()
    ref = float(np.sum(_np(x) ** 2))
    # contiguous input sums each 16-byte vector's squares in fp32 (at most 8
    # terms, each rounding within 2⁻²⁴) before the fp64 accumulation
    tol = 8 * 2.0**-24
    assert abs(out.item() - ref) <= tol * max(ref, 1e-300)
    # accumulate adds to the scalar; the order is fixed, so a repeat is bit-identical
    lg.logra_sum_squares(x, out, accumulate=True)
    torch.cuda.synchronize()
    assert abs(out.item() - 2 * ref) <= 2 * tol * max(ref, 1e-300)
    again = torch.zeros((1,), dtype=torch.float64, device=DEV)
    lg.logra_sum_squares(x, again)
    lg.logra_sum_squares(x, again, accumulate=True)
    torch.cuda.synchronize()
    assert again.item() == out.item()


@pytest.mark.parametrize("T,d,k,r,kind", [(300, 136, 520, 4, "signs"), (512, 256, 1536, 64, "signs"),
                                          (256, 64, 264, 256, "signs"), (200, 128, 1000, 16, "gauss")])
def test_reconstruction_cosine_matches_oracle(lg, T, d, k, r, kind):
    from rank_gradient_sketching_gb300.diagnostics import reconstruction_cosine

    seed, sid = 105, 3
    X, dY = synthetic.microbatch("tiny", 0, "rc", 0, T, d, k, DEV)
    if kind == "signs":
        got = reconstruction_cosine(X, dY, r, seed=seed, stream_id=sid)
        A = oph.projection(seed, sid, r, k)
    else:
        op = lg.logra_regen_projection(seed, sid, r, k, lg.LOGRA_PROJ_GAUSS_BF16)
        got = reconstruction_cosine(X, dY, r, operand=op)
        A = _np(op) / np.sqrt(r)  # the GPU's operand (its rounding is tested on its own)
    ref = odiag.reconstruction_cosine(_np(X), _np(dY), A)
    # the three norms on their own, against the same quantities in fp64
    from rank_gradient_sketching_gb300.diagnostics import reconstruction_terms

    s2, g2, r2 = reconstruction_terms(X, dY, r, seed=seed, stream_id=sid, operand=None if kind == "signs" else op)
    G = _np(dY).T @ _np(X)
    S = G @ A.T
    errs = (abs(s2 / np.sum(S * S) - 1), abs(g2 / np.sum(G * G) - 1), abs(r2 / np.sum((S @ A) ** 2) - 1))
    # ‖S‖² and ‖G‖² carry only fp32 accumulation and the hi/lo split of P;
    # S·A is rounded to bf16, each element within 2⁻⁹ of its value, so ‖S·A‖²
    # is within a factor (1 ± 2⁻⁹)² and the cosine within 1 ± 2⁻⁹
    assert errs[0] <= 1e-4 and errs[1] <= 1e-5
    assert errs[2] <= 2 * 2.0**-9 + 1e-5
    assert abs(got - ref) <= (2.0**-9 + 1e-4) * ref, errs


@pytest.mark.parametrize("r", [4, 64, 256])
def test_reconstruction_cosine_full_size_random_gradient(lg, r):
    # q projection of the 7B set, one 16384-token micro-batch: for inputs with
    # independent entries the cosine sits at tr(AAᵀ)/√(k·‖AAᵀ‖²) (close to
    # √(r/(r + k))), a value fixed by A alone
    from rank_gradient_sketching_gb300.diagnostics import reconstruction_cosine

    w = synthetic.WORKLOADS["qwen7b"]
    name, d, k, sid = [m for m in w["layers"][0] if m[0] == "q"][0]
    seed, T = w["seeds"][2], w["tokens"]
    X, dY = synthetic.microbatch("qwen7b", 2, name, 0, T, d, k, DEV)
    got = reconstruction_cosine(X, dY, r, seed=seed, stream_id=sid)
    A = oph.projection(seed, sid, r, k)
    AA = A @ A.T
    expect = np.trace(AA) / np.sqrt(k * np.sum(AA * AA))
    assert abs(got - expect) < 0.01 + 0.05 * expect
    assert abs(expect - np.sqrt(r / (r + k))) < 0.01
