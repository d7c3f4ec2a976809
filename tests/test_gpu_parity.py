"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances (the path's stated bounds): projection signs bit-exact; sketch S
within 1e-3 relative Frobenius error; merged bf16 weights within one bf16 ulp
of the oracle result (plus a 2⁻¹⁴ relative allowance on the update's
absolute-sum bound, for results that cancel to near zero); q(D) within 1e-4
relative.
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
    assert mod.logra_device_error() == 0
    yield mod
    assert mod.logra_device_error() == 0


DEV = "cuda"


def _np(t):
    return t.detach().double().cpu().numpy()


def _pad(t, mult=8):
    """The same values in a buffer whose row stride is a multiple of `mult`
    elements, as the ABI requires for 16-byte row alignment."""
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
    """How far inside the 1e-3 bound S lands: up to r = 64 P carries ~16
    significant bits (bf16 hi + lo), about 1e-5 in S; above, fp16 P carries
    11, about 2e-4 in S."""
    return 1e-4 if r <= 64 else 4e-4


# ---------------------------------------------------------------- projection

@pytest.mark.parametrize("seed,sid,r,k", [(0, 0, 4, 256), (1, 0, 64, 4096), ((1 << 40) + 5, 6, 256, 18944),
                                          (7, 3, 5, 300), (123, 4, 1, 1)])
def test_regen_signs_bit_exact(lg, seed, sid, r, k):
    got = lg.logra_regen_projection(seed, sid, r, k, lg.LOGRA_PROJ_INT8_PM1).cpu().numpy()
    assert np.array_equal(got, oph.signs(seed, sid, r, k))


def test_regen_scaled_outputs(lg):
    r, k = 64, 1000
    s = oph.signs(9, 2, r, k).astype(np.float64)
    f32 = lg.logra_regen_projection(9, 2, r, k, lg.LOGRA_PROJ_FP32).cpu().numpy()
    assert np.array_equal(f32, (s / 8.0).astype(np.float32))
    bf = lg.logra_regen_projection(9, 2, r, k, lg.LOGRA_PROJ_BF16).float().cpu().numpy()
    assert np.array_equal(bf, (s / 8.0).astype(np.float32))
    # padded row stride
    out = torch.zeros((5, 304), dtype=torch.int8, device=DEV)
    lg.logra_regen_projection(3, 1, 5, 300, lg.LOGRA_PROJ_INT8_PM1, out=out[:, :300])
    o = out.cpu().numpy()
    assert np.array_equal(o[:, :300], oph.signs(3, 1, 5, 300)) and np.all(o[:, 300:] == 0)


# -------------------------------------------------------------------- sketch

def _sketch_case(lg, T, d, k, r, nmb, seed=11, sid=2, s0=True, lds_pad=0, workload="tiny"):
    mbs = [tuple(_pad(t) for t in synthetic.microbatch(workload, 0, f"case{T}x{d}x{k}", m, T, d, k, DEV))
           for m in range(nmb)]
    S_full = torch.zeros((d, r + lds_pad), dtype=torch.float32, device=DEV)
    S = S_full[:, :r]
    if s0:
        S.copy_(torch.randn((d, r), generator=torch.Generator(device=DEV).manual_seed(5), device=DEV) * 1e-3)
    S0 = _np(S)
    ws = lg.sketch_workspace(T, d, k, r, DEV)
    for X, dY in mbs:
        lg.logra_sketch_accumulate(X, dY, S, seed, sid, r, ws)
    torch.cuda.synchronize()
    A = oph.projection(seed, sid, r, k)
    ref = osk.sketch_accumulate(S0, [(_np(X), _np(dY)) for X, dY in mbs], A)
    return _np(S), ref, mbs, ws


@pytest.mark.parametrize("T,d,k,r,nmb", [
    (128, 256, 256, 4, 2),       # the tiny single-layer workload
    (200, 136, 296, 5, 1),       # ragged against every tile size
    (77, 64, 64, 16, 1),         # less than one tile
    (1000, 304, 520, 100, 2),    # several tiles, r not a multiple of 16
    (512, 384, 640, 1, 1),
    (512, 384, 640, 16, 1),
    (512, 384, 640, 64, 1),
    (512, 384, 640, 256, 1),
    (4096, 256, 512, 64, 1),     # many split ranges of T
    (640, 1000, 200, 200, 1),
    (300, 136, 520, 250, 1),     # r just below the largest, ragged T, d and k
    (1, 8, 8, 1, 1),             # one token, the smallest matrix and rank
    (1, 8, 8, 256, 1),           # one token at the largest rank
])
def test_sketch_matches_oracle(lg, T, d, k, r, nmb):
    got, ref, _, _ = _sketch_case(lg, T, d, k, r, nmb)
    rel = _rel(got, ref)
    assert rel <= S_TOL, rel
    assert rel <= _tight(r), f"the sketch should be far inside the bound, got {rel}"


def test_sketch_padded_stride_and_zero_start(lg):
    got, ref, _, _ = _sketch_case(lg, 300, 200, 400, 24, 1, s0=False, lds_pad=8)
    assert _rel(got, ref) <= 1e-4


def test_sketch_never_reads_past_the_row_end(lg):
    # Row padding of X and dY holds NaN; the result must not see it.
    T, d, k, r = 300, 136, 200, 24
    X, dY = synthetic.microbatch("tiny", 0, "nanpad", 0, T, d, k, DEV)
    Xp = torch.full((T, k + 16), math.nan, dtype=torch.bfloat16, device=DEV)
    dYp = torch.full((T, d + 8), math.nan, dtype=torch.bfloat16, device=DEV)
    Xp[:, :k] = X
    dYp[:, :d] = dY
    S = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate(Xp[:, :k], dYp[:, :d], S, 6, 1, r)
    torch.cuda.synchronize()
    ref = osk.sketch_accumulate(np.zeros((d, r)), [(_np(X), _np(dY))], oph.projection(6, 1, r, k))
    assert torch.isfinite(S).all()
    assert _rel(_np(S), ref) <= 1e-4


def test_sketch_projection_intermediate(lg):
    # The workspace holds Pᵀ as bf16 hi + lo; together they must equal
    # X·(A√r)ᵀ to ~16 significant bits.
    T, d, k, r = 300, 128, 704, 20
    X, dY = synthetic.microbatch("tiny", 0, "inter", 0, T, d, k, DEV)
    S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
    ws = lg.sketch_workspace(T, d, k, r, DEV)
    lg.logra_sketch_accumulate(X, dY, S, 4, 1, r, ws)
    torch.cuda.synchronize()
    np16, Tp = 32, 384
    pb = (np16 * Tp * 2 + 255) // 256 * 256
    phi = ws[:np16 * Tp * 2].view(torch.bfloat16).view(np16, Tp)
    plo = ws[pb:pb + np16 * Tp * 2].view(torch.bfloat16).view(np16, Tp)
    P = (_np(phi) + _np(plo))[:r, :T].T
    P_ref = _np(X) @ oph.signs(4, 1, r, k).astype(np.float64).T
    assert _rel(P, P_ref) < 2e-5
    assert np.all(_np(phi)[r:] == 0) and np.all(_np(plo)[r:] == 0)
    assert np.all(_np(phi)[:, T:] == 0)


def test_sketch_p16_intermediate(lg):
    # Above r = 64 the workspace holds Pᵀ as fp16 scaled per group of 16
    # tokens, and the token scales g_t = 2^e_t: powers of two, equal within a
    # group, that put the group's largest |P| in [2^14, 2^15) before rounding,
    # with P16·g equal to X·(A√r)ᵀ to fp16 precision.  The tokens' magnitudes
    # swing over 2^40 here, so a group holds tokens 2^15 apart.
    T, d, k, r = 300, 128, 704, 100
    X, dY = synthetic.microbatch("tiny", 0, "inter16", 0, T, d, k, DEV)
    X = X * torch.exp2(torch.arange(T, device=DEV).float().remainder(41) - 20)[:, None].to(torch.bfloat16)
    S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
    ws = lg.sketch_workspace(T, d, k, r, DEV)
    lg.logra_sketch_accumulate(X, dY, S, 4, 1, r, ws)
    torch.cuda.synchronize()
    np16, Tp = 112, 384
    # blocks of 64 tokens, each two halves (one per CTA of a contraction pair):
    # 64 fp32 token scales, then np16/2 rows of 64 fp16 tokens under the
    # 128-byte swizzle (16-byte chunk c of local row n stored at chunk c ^ (n & 7))
    hn, hb = np16 // 2, 256 + np16 * 64
    raw = ws[:(Tp // 64) * 2 * hb].cpu().numpy().reshape(Tp // 64, 2, hb)
    g = raw[:, 0, :256].copy().view(np.float32).reshape(-1).astype(np.float64)
    assert np.array_equal(raw[:, 0, :256], raw[:, 1, :256])          # both halves carry the scales
    rows = raw[:, :, 256:].copy().view(np.float16).reshape(Tp // 64, 2, hn, 8, 8).astype(np.float64)
    nl = np.arange(hn)[:, None]
    src_chunk = np.arange(8)[None, :] ^ (nl & 7)
    p16 = np.concatenate([np.concatenate([rows[b, h][nl, src_chunk].reshape(hn, 64) for b in range(Tp // 64)], axis=1)
                          for h in range(2)], axis=0)
    m, e = np.frexp(g[:T])
    assert np.all(m == 0.5)                                   # powers of two
    gg = g[:Tp].reshape(-1, 16)
    assert np.all(gg == gg[:, :1])                            # one scale per 16-token group
    top = np.abs(p16[:r, :T]).max(axis=0)
    top = np.array([top[j:j + 16].max() for j in range(0, T, 16)])
    # (a maximum just under 2^15 may round up to 2^15 itself: fp16 spacing is 16 there)
    assert np.all((top >= 2.0**14) & (top <= 2.0**15))
    P = (p16[:r, :T] * g[:T]).T
    P_ref = _np(X) @ oph.signs(4, 1, r, k).astype(np.float64).T
    assert _rel(P, P_ref) < 3e-4
    assert np.all(p16[r:] == 0) and np.all(p16[:, T:] == 0)
    ref = osk.sketch_accumulate(np.zeros((d, r)), [(_np(X), _np(dY))], oph.projection(4, 1, r, k))
    assert _rel(_np(S), ref) <= _tight(r)


def _row_rel(a, b):
    return np.linalg.norm(a - b, axis=1) / np.linalg.norm(b, axis=1)


@pytest.mark.parametrize("d,r", [(256, 128), (8192, 128), (1024, 256)])
def test_sketch_p16_row_scales_follow_each_row(lg, d, r):
    # dY rows whose magnitude moves far more than fp16's range along T: rows
    # that grow by 2^64 over the tokens, rows that shrink by as much, rows that
    # are zero for the first half and then tiny (1e-20), rows with one spike of
    # 1e30; X rows whose scale swings over 2^±20.  Each row of S must still be
    # within the bound on its own (a Frobenius check over all of S would be
    # blind to the small rows).  With d = 8192 a contraction CTA covers all
    # 2048 tokens (one split), so its rows lower their scale several times.
    T, k = 2048, 256
    g = torch.Generator(device=DEV).manual_seed(d + r)
    X = torch.randn((T, k), generator=g, device=DEV)
    X = (X * torch.exp2(torch.arange(T, device=DEV).float().remainder(41) - 20)[:, None]).to(torch.bfloat16)
    base = torch.randn((T, d), generator=g, device=DEV)
    t = torch.arange(T, device=DEV).float()[:, None]
    q = d // 4
    dY = torch.empty((T, d), device=DEV)
    dY[:, :q] = base[:, :q] * torch.exp2(t / 32)
    dY[:, q:2 * q] = base[:, q:2 * q] * torch.exp2(-t / 32)
    dY[:, 2 * q:3 * q] = torch.where(t < 1000, torch.zeros_like(base[:, 2 * q:3 * q]), base[:, 2 * q:3 * q] * 1e-20)
    dY[:, 3 * q:] = base[:, 3 * q:]
    dY[1500, 3 * q:] = 1e30
    dY = dY.to(torch.bfloat16)
    S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
    lg.logra_sketch_accumulate(X, dY, S, 9, 3, r)
    torch.cuda.synchronize()
    if d == 8192:
        assert lg.logra_sketch_splits(T, d, k, r) == 1
    ref = osk.sketch_accumulate(np.zeros((d, r)), [(_np(X), _np(dY))], oph.projection(9, 3, r, k))
    got = _np(S)
    assert np.all(np.isfinite(got))
    rel = _row_rel(got, ref)
    assert rel.max() <= S_TOL, (rel.argmax(), rel.max())
    assert np.median(rel) <= _tight(r)


def test_sketch_bitwise_deterministic(lg):
    T, d, k, r = 2048, 256, 384, 64
    X, dY = synthetic.microbatch("tiny", 0, "det", 0, T, d, k, DEV)
    outs = []
    for _ in range(3):
        S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
        lg.logra_sketch_accumulate(X, dY, S, 1, 0, r)
        outs.append(S.clone())
    assert lg.logra_sketch_splits(T, d, k, r) > 1
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_sketch_p16_bitwise_deterministic(lg):
    # the fp16 contraction with split ranges (and a row scale lowered mid-way)
    T, d, k, r = 2048, 256, 384, 256
    X, dY = synthetic.microbatch("tiny", 0, "det16", 0, T, d, k, DEV)
    dY = (dY.float() * torch.exp2(torch.arange(T, device=DEV).float() / 64)[:, None]).to(torch.bfloat16)
    outs = []
    for _ in range(3):
        S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
        lg.logra_sketch_accumulate(X, dY, S, 1, 0, r)
        outs.append(S.clone())
    assert lg.logra_sketch_splits(T, d, k, r) > 1
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_sketch_linear_in_microbatches(lg):
    T, d, k, r = 256, 128, 256, 16
    (X1, dY1), (X2, dY2) = [synthetic.microbatch("tiny", 0, "lin", m, T, d, k, DEV) for m in range(2)]
    S_a = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate(X1, dY1, S_a, 3, 0, r)
    lg.logra_sketch_accumulate(X2, dY2, S_a, 3, 0, r)
    S_b = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate(torch.cat([X1, X2]), torch.cat([dY1, dY2]), S_b, 3, 0, r)
    torch.cuda.synchronize()
    assert _rel(_np(S_a), _np(S_b)) < 1e-5


def _sampled_rows_check(lg, workload, T, d, k, r, nmb, seed, sid, rows):
    mbs_dev = [synthetic.microbatch(workload, 0, f"full{d}x{k}", m, T, d, k, DEV) for m in range(nmb)]
    S = torch.zeros((d, r), dtype=torch.float32, device=DEV)
    ws = lg.sketch_workspace(T, d, k, r, DEV)
    for X, dY in mbs_dev:
        lg.logra_sketch_accumulate(X, dY, S, seed, sid, r, ws)
    torch.cuda.synchronize()
    A = oph.projection(seed, sid, r, k)
    mbs = [(_np(X), _np(dY[:, rows])) for X, dY in mbs_dev]
    ref = osk.sketch_rows(np.zeros((len(rows), r)), np.arange(len(rows)), mbs, A)
    got = _np(S)[rows]
    assert _rel(got, ref) <= S_TOL
    assert _rel(got, ref) <= _tight(r)
    # all rows finite, and rows outside the sample are not all zero
    assert torch.isfinite(S).all()


def test_sketch_square_workload_sampled_rows(lg):
    # d = k = 4096, r = 64, 8 micro-batches of 4096 tokens, projection seed 1
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 3000, 4095])
    _sampled_rows_check(lg, "square", 4096, 4096, 4096, 64, 8, 1, 0, rows)


@pytest.mark.parametrize("d,k,r", [(18944, 3584, 256), (3584, 18944, 64), (512, 3584, 256), (8960, 1536, 16)])
def test_sketch_qwen_matrices_sampled_rows(lg, d, k, r):
    # full-size single matrices of the 7B / 1.5B projection sets, one micro-batch
    T = 16384 if k == 3584 or d == 3584 else 8192
    rng = np.random.default_rng(d + k)
    rows = np.unique(np.concatenate([[0, d - 1], rng.integers(0, d, 10)]))
    _sampled_rows_check(lg, "qwen7b" if T == 16384 else "qwen1.5b", T, d, k, r, 1, 113, 4, rows)


# --------------------------------------------------------------------- merge

def _merge_check(lg, d, k, r, ae, seed=21, sid=5, use_dev_scalar=False, ldw_pad=0):
    Wf = torch.zeros((d, k + ldw_pad), dtype=torch.bfloat16, device=DEV)
    W = Wf[:, :k]
    W.copy_(synthetic.weight("tiny", 0, f"m{d}x{k}", d, k, DEV))
    if ldw_pad == 0 and k % 8:
        W = _pad(W)
        Wf = W.as_strided((d, W.stride(0)), (W.stride(0), 1))
    S = torch.randn((d, r), generator=torch.Generator(device=DEV).manual_seed(d * r), device=DEV) * 0.15
    W0 = _np(W)
    pad0 = Wf[:, k:].clone()
    if use_dev_scalar:
        lg.logra_merge_update(W, S, seed, sid, r, 123.0, alpha_eta_dev=torch.tensor(ae, dtype=torch.float32,
                                                                                    device=DEV))
    else:
        lg.logra_merge_update(W, S, seed, sid, r, ae)
    torch.cuda.synchronize()
    A = oph.projection(seed, sid, r, k)
    ae32 = float(np.float32(ae))
    ref = omerge.merge(W0, _np(S), A, ae32)
    got = _np(W)
    n_allow = merge_check(got, ref, W0, _np(S), A, ae32, what=f"merge {d}x{k} r={r}")
    assert torch.equal(Wf[:, k:], pad0)  # bytes past k are untouched
    return got, ref, W0, n_allow


@pytest.mark.parametrize("d,k,r", [(256, 256, 4), (300, 520, 5), (100, 72, 1), (256, 256, 8), (256, 256, 16),
                                   (384, 1000, 64), (130, 200, 100), (256, 512, 256), (129, 72, 9),
                                   # above r = 128 row tiles go in clusters of two: an odd tile
                                   # count (3, and 1) adds a padding tile past d
                                   (300, 520, 200), (100, 72, 144), (129, 1000, 256)])
def test_merge_matches_oracle(lg, d, k, r):
    _merge_check(lg, d, k, r, 1e-3)


def test_merge_square_workload(lg):
    got, ref, W0, n_allow = _merge_check(lg, 4096, 4096, 64, 2e-4)
    print(f"[merge tolerance] square 4096x4096 r=64: {n_allow} of {got.size} weights outside a strict 1-ulp "
          "bound, all cancellations")
    assert n_allow <= 4 + 2 * got.size // 10**6
    assert np.mean(got != W0) > 0.01  # the update actually changed weights


@pytest.mark.parametrize("r", [4, 40])
def test_merge_leaves_row_padding_alone(lg, r):
    d, k = 130, 264
    Wp = torch.full((d, k + 8), math.nan, dtype=torch.bfloat16, device=DEV)
    Wp[:, :k] = synthetic.weight("tiny", 0, "pad", d, k, DEV)
    S = torch.randn((d, r), generator=torch.Generator(device=DEV).manual_seed(r), device=DEV)
    lg.logra_merge_update(Wp[:, :k], S, 1, 2, r, 1e-3)
    torch.cuda.synchronize()
    assert torch.isnan(Wp[:, k:].float()).all()
    assert torch.isfinite(Wp[:, :k].float()).all()


def test_merge_zero_step_bit_exact(lg):
    for r in (4, 64):
        W = synthetic.weight("tiny", 0, "z", 200, 304, DEV)
        W0 = W.clone()
        S = torch.randn((200, r), device=DEV)
        lg.logra_merge_update(W, S, 1, 1, r, 0.0)
        torch.cuda.synchronize()
        assert torch.equal(W, W0)


def test_merge_device_scalar_and_padded_stride(lg):
    _merge_check(lg, 200, 296, 4, 5e-3, use_dev_scalar=True, ldw_pad=8)
    _merge_check(lg, 200, 296, 40, 5e-3, use_dev_scalar=True, ldw_pad=8)


def test_merge_single_entry_closed_form(lg):
    d, k, r = 64, 384, 32
    W = synthetic.weight("tiny", 0, "one", d, k, DEV)
    W0 = _np(W)
    S = torch.zeros((d, r), device=DEV)
    S[7, 13] = 0.5
    lg.logra_merge_update(W, S, 2, 3, r, 0.25)
    torch.cuda.synchronize()
    got = _np(W)
    sign = oph.signs(2, 3, r, k)[13].astype(np.float64)
    row = omerge.bf16_round(W0[7] - 0.25 * 0.5 * sign / math.sqrt(r))
    assert np.array_equal(got[7], row)
    assert np.array_equal(np.delete(got, 7, 0), np.delete(W0, 7, 0))


# ------------------------------------------------------------------------ KL

def _kl_check(lg, cur, prop, tau=1.0, mask=None):
    row_kl = torch.empty(cur.shape[0], dtype=torch.float32, device=DEV)
    q = lg.logra_predicted_kl(cur, prop, tau, row_mask=mask, row_kl_out=row_kl)
    torch.cuda.synchronize()
    q_ref, kl_ref = okl.predicted_kl(_np(cur), _np(prop), tau, None if mask is None else mask.cpu().numpy())
    return float(q.item()), q_ref, row_kl.double().cpu().numpy(), kl_ref


def test_kl_tiny_workload(lg):
    cur, prop = synthetic.kl_logits("tiny", 0.05, device=DEV)
    q, q_ref, rk, rk_ref = _kl_check(lg, cur, prop)
    assert abs(q - q_ref) <= Q_TOL * q_ref
    assert np.allclose(rk, rk_ref, rtol=Q_TOL, atol=0)


@pytest.mark.parametrize("eps", [0.01, 0.1])
def test_kl_qwen_rows(lg, eps):
    # 64 rows of the full-vocabulary bf16 workload (boosted entries included)
    cur, prop = synthetic.kl_logits("qwen", eps, rows=64, device=DEV)
    q, q_ref, rk, rk_ref = _kl_check(lg, cur, prop)
    assert abs(q - q_ref) <= Q_TOL * q_ref, (q, q_ref)
    assert np.allclose(rk, rk_ref, rtol=Q_TOL, atol=0)


@pytest.mark.parametrize("dtype,V,tau", [(torch.float32, 1001, 1.0), (torch.bfloat16, 1001, 0.7),
                                         (torch.bfloat16, 7, 1.0), (torch.float32, 5000, 2.0)])
def test_kl_ragged_vocab_and_temperature(lg, dtype, V, tau):
    g = torch.Generator(device=DEV).manual_seed(V)
    a = _pad((torch.randn((9, V), generator=g, device=DEV) * 3).to(dtype))
    b = _pad((a.float() + 0.3 * torch.randn((9, V), generator=g, device=DEV)).to(dtype))
    q, q_ref, rk, rk_ref = _kl_check(lg, a, b, tau)
    assert abs(q - q_ref) <= Q_TOL * q_ref
    assert np.allclose(rk, rk_ref, rtol=Q_TOL, atol=0)


def test_kl_large_differences_and_padded_rows(lg):
    g = torch.Generator(device=DEV).manual_seed(3)
    full_a = torch.zeros((6, 2056), device=DEV)
    full_b = torch.zeros((6, 2056), device=DEV)
    full_a[:, :2050] = torch.randn((6, 2050), generator=g, device=DEV) * 2
    full_b[:, :2050] = full_a[:, :2050] + torch.randn((6, 2050), generator=g, device=DEV) * 2.5
    q, q_ref, rk, rk_ref = _kl_check(lg, full_a[:, :2050], full_b[:, :2050])
    assert abs(q - q_ref) <= Q_TOL * q_ref
    assert np.allclose(rk, rk_ref, rtol=Q_TOL, atol=0)


def test_kl_unchanged_model_is_zero(lg):
    cur, _ = synthetic.kl_logits("tiny", 0.05, device=DEV)
    q, q_ref, rk, _ = _kl_check(lg, cur, cur.clone())
    assert q == 0.0 and q_ref == 0.0 and np.all(rk == 0.0)


def test_kl_infinities_nan_and_mask(lg):
    a = torch.randn((4, 64), generator=torch.Generator(device=DEV).manual_seed(1), device=DEV)
    b = a + 0.1
    b[:, 5] += 0.7
    a[0, 3] = -math.inf          # p = 0: no contribution
    b[0, 3] = 5.0
    b[1, 9] = -math.inf          # finite p, p' = 0: +inf
    a[2, 11] = math.nan          # NaN propagates
    mask = torch.tensor([1, 0, 0, 1], dtype=torch.uint8, device=DEV)
    q, q_ref, rk, rk_ref = _kl_check(lg, a, b, mask=mask)
    assert abs(rk[0] - rk_ref[0]) <= Q_TOL * rk_ref[0]
    assert rk[1] == math.inf and rk_ref[1] == math.inf
    assert math.isnan(rk[2]) and math.isnan(rk_ref[2])
    assert abs(rk[3] - rk_ref[3]) <= Q_TOL * rk_ref[3]
    assert abs(q - q_ref) <= Q_TOL * q_ref
    none = torch.zeros(4, dtype=torch.uint8, device=DEV)
    assert float(lg.logra_predicted_kl(a, b, 1.0, row_mask=none).item()) == 0.0
    empty = torch.empty((0, 64), device=DEV)
    assert float(lg.logra_predicted_kl(empty, empty, 1.0).item()) == 0.0


def test_kl_quadratic_model(lg):
    # halving the step quarters the predicted KL (the controller's model)
    g = torch.Generator(device=DEV).manual_seed(8)
    a = torch.randn((32, 4096), generator=g, device=DEV) * 3
    delta = torch.randn((32, 4096), generator=g, device=DEV)
    q1 = float(lg.logra_predicted_kl(a, a + 2e-2 * delta).item())
    q2 = float(lg.logra_predicted_kl(a, a + 1e-2 * delta).item())
    assert abs(q2 / q1 - 0.25) < 0.01


def test_step_size_device_matches_oracle(lg):
    for q in [0.0, 1e-7, 8e-4, 3.0]:
        q_dev = torch.tensor(q, dtype=torch.float64, device=DEV)
        ae = torch.empty((), dtype=torch.float32, device=DEV)
        al = torch.empty((), dtype=torch.float64, device=DEV)
        lg.logra_step_size_device(q_dev, 2e-4, 1.0, 1e-3, ae, al)
        a_ref = ostep.step_size(q, 2e-4, 1.0)
        assert float(al.item()) == a_ref
        assert float(ae.item()) == float(np.float32(a_ref * 1e-3))


@pytest.mark.parametrize("r", [16, 64, 200, 256])
def test_merge_s_row_strides(lg, r):
    # S with row stride r or r + 4 is staged by TMA, r + 1 takes the loaded
    # path; the three must give the same weights bit for bit
    d, k, ae = 300, 520, 3e-3
    base = torch.randn((d, r), generator=torch.Generator(device=DEV).manual_seed(r), device=DEV) * 0.1
    outs = []
    for pad in (0, 4, 1):
        Sb = torch.zeros((d, r + pad), device=DEV)
        Sb[:, :r] = base
        W = synthetic.weight("tiny", 0, "ms", d, k, DEV)
        lg.logra_merge_update(W, Sb[:, :r], 9, 4, r, ae)
        outs.append(W)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    W0 = _np(synthetic.weight("tiny", 0, "ms", d, k, DEV))
    A = oph.projection(9, 4, r, k)
    ref = omerge.merge(W0, _np(base), A, float(np.float32(ae)))
    merge_check(_np(outs[0]), ref, W0, _np(base), A, float(np.float32(ae)))
