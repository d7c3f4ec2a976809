"""Pins of the fp64 oracle against facts fixed outside the oracle itself:
published known-answer vectors, the page's worked examples, closed forms,
library routines and brute force on tiny inputs.  CPU only."""

import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp, rel_entr

from oracle import kl as okl
from oracle import merge as omerge
from oracle import philox as oph
from oracle import sketch as osk
from oracle import step as ostep

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_kv(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


# --------------------------------------------------------------------- Philox

def test_philox_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for row in rows:
        v = [int(x, 16) for x in row]
        out = oph.philox4x32_10(np.array(v[0:4], dtype=np.uint64), np.array(v[4:6], dtype=np.uint64))
        assert [int(x) for x in out] == v[6:10]


def test_philox_vectorised_matches_single_calls():
    rng = np.random.default_rng(3)
    ctr = rng.integers(0, 2**32, size=(7, 4), dtype=np.uint64)
    key = rng.integers(0, 2**32, size=(7, 2), dtype=np.uint64)
    batch = oph.philox4x32_10(ctr, key)
    for i in range(7):
        assert np.array_equal(batch[i], oph.philox4x32_10(ctr[i], key[i]))


def test_sign_stream_prefix_and_independence():
    a = oph.sign_bits(11, 3, 6, 1000)
    # columns and rows are prefixes of the same stream, whatever r and k are
    assert np.array_equal(oph.sign_bits(11, 3, 6, 300), a[:, :300])
    assert np.array_equal(oph.sign_bits(11, 3, 2, 1000), a[:2])
    # another stream id or seed gives another stream
    assert (oph.sign_bits(11, 4, 6, 1000) != a).mean() > 0.4
    assert (oph.sign_bits(12, 3, 6, 1000) != a).mean() > 0.4
    # 64-bit seeds: the high word matters
    assert (oph.sign_bits(11 + (1 << 32), 3, 6, 1000) != a).mean() > 0.4


def test_sign_stream_word_layout():
    # column j of row i is bit (j & 31) of word (j & 127) >> 5 of the call with
    # counter (j >> 7, i, stream, 0): check a few columns against single calls
    seed, sid = 0x1234_5678_9ABC, 9
    bits = oph.sign_bits(seed, sid, 5, 777)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint64)
    for i, j in [(0, 0), (4, 31), (2, 32), (3, 127), (1, 128), (4, 776)]:
        w = oph.philox4x32_10(np.array([j >> 7, i, sid, 0], dtype=np.uint64), key)
        assert bits[i, j] == (int(w[(j & 127) >> 5]) >> (j & 31)) & 1


@pytest.mark.parametrize("r", [4, 16, 64, 256])
def test_projection_gram_diagonal_exact_and_balance(r):
    k = 512
    A = oph.projection(7, 0, r, k)
    G = A.T @ A
    assert np.all(np.diag(G) == 1.0)  # Σ_i (±1/√r)² = 1 exactly
    off = G[~np.eye(k, dtype=bool)]
    assert abs(off.mean()) < 5 / math.sqrt(r * off.size) + 1e-3
    assert abs(off.std() - 1 / math.sqrt(r)) < 0.05 / math.sqrt(r)
    frac = oph.sign_bits(7, 0, r, k).mean()
    assert abs(frac - 0.5) < 5 * 0.5 / math.sqrt(r * k)


def test_projection_expected_gram_is_identity():
    r, k, n = 4, 24, 3000
    acc = np.zeros((k, k))
    for s in range(n):
        A = oph.projection(s, 0, r, k)
        acc += A.T @ A
    acc /= n
    assert np.allclose(acc, np.eye(k), atol=5 / math.sqrt(n * r))


# --------------------------------------------------------------------- sketch

def _bf16_values(shape, std, seed):
    t = torch.randn(shape, generator=torch.Generator().manual_seed(seed)) * std
    return t.to(torch.bfloat16).double().numpy()


def test_sketch_equals_projected_inputs_brute_force():
    # all dimensions distinct so that a transposed operand cannot pass
    T, d, k, r = 5, 3, 7, 2
    X = _bf16_values((T, k), 1.0, 1)
    dY = _bf16_values((T, d), 1.0, 2)
    A = oph.projection(5, 1, r, k)
    S0 = _bf16_values((d, r), 1.0, 3)
    ref = [[S0[i][j] for j in range(r)] for i in range(d)]
    for i in range(d):
        for j in range(r):
            for t in range(T):
                p = 0.0
                for l in range(k):
                    p += X[t][l] * A[j][l]
                ref[i][j] += dY[t][i] * p
    got = osk.sketch_accumulate(S0, [(X, dY)], A)
    assert np.allclose(got, np.array(ref), rtol=1e-12, atol=1e-12)


def test_sketch_linear_across_microbatches():
    T, d, k, r = 9, 6, 10, 4
    A = oph.projection(2, 0, r, k)
    mbs = [(_bf16_values((T, k), 1.0, 10 + m), _bf16_values((T, d), 1e-3, 20 + m)) for m in range(3)]
    S0 = np.zeros((d, r))
    whole = osk.sketch_accumulate(S0, mbs, A)
    parts = sum(osk.sketch_accumulate(S0, [mb], A) for mb in mbs)
    assert np.allclose(whole, parts, rtol=1e-12, atol=1e-15)
    # and a dropped micro-batch is visible
    assert not np.allclose(whole, osk.sketch_accumulate(S0, mbs[:2], A), rtol=1e-6)
    # concatenating the micro-batches along T is the same as accumulating them
    Xc = np.concatenate([m[0] for m in mbs])
    dYc = np.concatenate([m[1] for m in mbs])
    assert np.allclose(whole, osk.sketch_accumulate(S0, [(Xc, dYc)], A), rtol=1e-12, atol=1e-15)


def test_sketch_rows_match_full():
    T, d, k, r = 8, 12, 9, 3
    A = oph.projection(4, 2, r, k)
    mbs = [(_bf16_values((T, k), 1.0, 30), _bf16_values((T, d), 1.0, 31))]
    S0 = _bf16_values((d, r), 1.0, 32)
    full = osk.sketch_accumulate(S0, mbs, A)
    rows = [0, 5, 11]
    assert np.allclose(osk.sketch_rows(S0[rows], rows, mbs, A), full[rows], rtol=1e-13)


def test_page_memory_example():
    g = _golden_kv("page_examples.txt")
    full, sk = osk.accumulator_bytes(int(g["memory.d"]), int(g["memory.k"]), int(g["memory.r"]), 4)
    assert full == g["memory.full_MiB"] * 2**20
    assert sk == g["memory.sketch_MiB"] * 2**20


# ---------------------------------------------------------------------- merge

def test_bf16_round_hand_worked():
    cases = {
        1.0 + 2**-8: 1.0,                  # tie between 1 and 1+2^-7 → even (1)
        1.0 + 3 * 2**-8: 1.0 + 2**-6,      # tie between 1+2^-7 and 1+2^-6 → even
        1.0 + 2**-8 + 2**-30: 1.0 + 2**-7,  # just above the tie
        -(1.0 + 3 * 2**-8): -(1.0 + 2**-6),
        2**-133: 2**-133,                  # smallest bf16 subnormal
        2**-134: 0.0,                      # tie to even (zero)
        3 * 2**-134: 2**-132,              # tie between 1 and 2 subnormal units → 2
        3.4e38: math.inf,                  # above the bf16 maximum
        0.1: 0.10009765625,
    }
    for x, want in cases.items():
        assert omerge.bf16_round(np.array([x]))[0] == want, x
    z = omerge.bf16_round(np.array([-0.0, -1e-50]))
    assert np.all(z == 0) and np.all(np.signbit(z))
    assert np.isnan(omerge.bf16_round(np.array([np.nan]))[0])


def test_bf16_round_matches_torch_on_fp32_inputs():
    x = torch.randn(200000, generator=torch.Generator().manual_seed(0)) * torch.logspace(-30, 30, 200000)
    want = x.to(torch.bfloat16).double().numpy()
    got = omerge.bf16_round(x.double().numpy())
    assert np.array_equal(got, want)


def test_bf16_ulp():
    assert omerge.bf16_ulp(np.array([1.0]))[0] == 2**-7
    assert omerge.bf16_ulp(np.array([1.99]))[0] == 2**-7
    assert omerge.bf16_ulp(np.array([2.0]))[0] == 2**-6
    assert omerge.bf16_ulp(np.array([0.02]))[0] == 2**-13


def test_merge_zero_step_is_identity():
    d, k, r = 6, 40, 4
    W = _bf16_values((d, k), 0.02, 40)
    S = _bf16_values((d, r), 1.0, 41)
    A = oph.projection(0, 0, r, k)
    assert np.array_equal(omerge.merge(W, S, A, 0.0), W)


def test_merge_single_entry_closed_form():
    d, k, r = 5, 300, 8
    W = _bf16_values((d, k), 0.02, 42)
    A = oph.projection(3, 1, r, k)
    S = np.zeros((d, r))
    i, n, s, ae = 2, 5, 0.75, 1e-2
    S[i, n] = s
    got = omerge.merge(W, S, A, ae)
    sign = oph.signs(3, 1, r, k)[n].astype(np.float64)
    row = W[i] - ae * s * sign / math.sqrt(r)
    assert np.array_equal(got[i], omerge.bf16_round(row))
    others = [x for x in range(d) if x != i]
    assert np.array_equal(got[others], W[others])
    # the sign matters: W − u, not W + u
    assert not np.array_equal(got[i], omerge.bf16_round(W[i] + ae * s * sign / math.sqrt(r)))


# ------------------------------------------------------------------------- KL

def test_kl_nonnegative_and_zero_for_unchanged():
    a = _bf16_values((20, 300), 3.0, 50)
    b = a + _bf16_values((20, 300), 0.1, 51)
    _, kl = okl.predicted_kl(a, b, 1.0)
    assert np.all(kl >= 0)
    q0, kl0 = okl.predicted_kl(a, a.copy(), 1.0)
    assert q0 == 0.0 and np.all(kl0 == 0.0)


def test_kl_two_token_closed_form():
    for a0, a1, b0, b1 in [(0.0, 1.0, 0.3, -0.2), (5.0, -5.0, 4.0, -4.5), (2.0, 2.0, 0.0, 1.0)]:
        p1 = expit(a1 - a0)
        q1 = expit(b1 - b0)
        want = (1 - p1) * math.log((1 - p1) / (1 - q1)) + p1 * math.log(p1 / q1)
        _, kl = okl.predicted_kl(np.array([[a0, a1]]), np.array([[b0, b1]]), 1.0)
        assert abs(kl[0] - want) <= 1e-12 * max(1.0, abs(want))
        # the direction is KL(current ‖ proposed)
        if a0 != a1 or b0 != b1:
            rev = p1 * 0 + (1 - q1) * math.log((1 - q1) / (1 - p1)) + q1 * math.log(q1 / p1)
            if abs(rev - want) > 1e-6:
                assert abs(kl[0] - rev) > 1e-7


def test_kl_uniform_current_closed_form():
    V = 1000
    b = _bf16_values((3, V), 2.0, 52)
    a = np.zeros((3, V))
    _, kl = okl.predicted_kl(a, b, 1.0)
    want = logsumexp(b, axis=1) - b.mean(axis=1) - math.log(V)
    assert np.allclose(kl, want, rtol=1e-12)


def test_kl_matches_scipy_rel_entr_and_temperature():
    a = _bf16_values((6, 500), 3.0, 53)
    b = a + _bf16_values((6, 500), 0.5, 54)
    tau = 0.7
    p = np.exp(a / tau - logsumexp(a / tau, axis=1, keepdims=True))
    q = np.exp(b / tau - logsumexp(b / tau, axis=1, keepdims=True))
    want = rel_entr(p, q).sum(axis=1)
    _, kl = okl.predicted_kl(a, b, tau)
    assert np.allclose(kl, want, rtol=1e-10)
    _, kl1 = okl.predicted_kl(a / tau, b / tau, 1.0)
    assert np.allclose(kl, kl1, rtol=1e-12)


def test_kl_quadratic_in_step():
    # the page's quadratic model: predicted KL of a + αΔ scales as α²
    a = _bf16_values((8, 400), 3.0, 55)
    delta = _bf16_values((8, 400), 1.0, 56)
    alpha = 1e-3
    q1, _ = okl.predicted_kl(a, a + alpha * delta, 1.0)
    q2, _ = okl.predicted_kl(a, a + 0.5 * alpha * delta, 1.0)
    assert abs(q2 / q1 - 0.25) < 1e-2


def test_kl_infinite_logits_and_mask():
    a = np.array([[0.0, 1.0, -np.inf], [0.0, 1.0, 2.0]])
    b = np.array([[0.5, 0.0, 3.0], [0.5, 0.0, -np.inf]])
    _, kl = okl.predicted_kl(a, b, 1.0)
    # row 0: the −inf current logit has p = 0 and drops out (prop renormalises)
    _, ref = okl.predicted_kl(a[:1, :2], np.array([[0.5, 0.0]]) , 1.0)
    p = np.exp(a[0, :2] - logsumexp(a[0, :2]))
    lq = b[0] - logsumexp(b[0])
    assert abs(kl[0] - np.sum(p * (np.log(p) - lq[:2]))) < 1e-12
    assert kl[1] == np.inf
    q, _ = okl.predicted_kl(a, b, 1.0, row_mask=np.array([1, 0], dtype=np.uint8))
    assert q == kl[0]
    q_none, _ = okl.predicted_kl(a, b, 1.0, row_mask=np.array([0, 0], dtype=np.uint8))
    assert q_none == 0.0
    _, kln = okl.predicted_kl(np.array([[0.0, np.nan]]), np.array([[0.0, 1.0]]), 1.0)
    assert np.isnan(kln[0])


# ----------------------------------------------------------------------- step

def test_step_size_page_example_and_cap():
    g = _golden_kv("page_examples.txt")
    delta = 2e-4
    assert ostep.step_size(g["controller.q_over_delta"] * delta, delta, 1.0) == g["controller.alpha"]
    assert ostep.step_size(g["controller.q_over_delta"] * delta, delta, 0.3) == 0.3
    assert ostep.step_size(0.0, delta, 0.8) == 0.8
    assert ostep.step_size(-1e-12, delta, 0.8) == 0.8
    assert math.isnan(ostep.step_size(math.nan, delta, 1.0))
    assert ostep.step_size(math.inf, delta, 1.0) == 0.0
    # halving α quarters the predicted KL α²·q
    q = 3e-3
    alpha = ostep.step_size(q, delta, 1.0)
    assert math.isclose((alpha / 2) ** 2 * q / (alpha**2 * q), g["controller.halving_factor"])
    # the controller hits the budget exactly when not capped: α²·q = δ
    assert math.isclose(alpha**2 * q, delta, rel_tol=1e-14)


def test_delta_schedule():
    s = ostep.delta_schedule(2e-4, 2e-5, 10)
    assert len(s) == 10 and s[0] == 2e-4 and math.isclose(s[-1], 2e-5)
    assert np.all(np.diff(s) < 0)
    assert np.allclose(np.diff(s), np.diff(s)[0])


# ---------------------------------------------------------------- momentum
def test_momentum_special_cases_and_closed_forms():
    from oracle import momentum as omom

    rng = np.random.default_rng(7)
    Ss = [rng.standard_normal((5, 3)) for _ in range(6)]
    # β = 0: the plain update U = S of the page
    assert np.array_equal(omom.momentum_run(Ss, 0.0), Ss[-1])
    # β = 1: the sum of the sketches
    assert np.allclose(omom.momentum_run(Ss, 1.0), np.sum(Ss, axis=0), rtol=1e-14, atol=0)
    # constant S: geometric series S·(1 − βⁿ)/(1 − β)
    beta, n = 0.9, 7
    S = rng.standard_normal((4, 2))
    assert np.allclose(omom.momentum_run([S] * n, beta), S * (1 - beta**n) / (1 - beta), rtol=1e-13, atol=0)
    # unrolled: M_n = Σ_t β^(n−t) S_t (catches dampening, or β applied to S)
    b = 0.75
    unrolled = sum(b ** (len(Ss) - 1 - t) * Ss[t] for t in range(len(Ss)))
    assert np.allclose(omom.momentum_run(Ss, b), unrolled, rtol=1e-13, atol=1e-15)
    # linear in the sketches
    assert np.allclose(omom.momentum_run([3.0 * s for s in Ss], b), 3.0 * omom.momentum_run(Ss, b), rtol=1e-13)
    with pytest.raises(ValueError):
        omom.momentum_update(np.zeros((2, 2)), np.zeros((2, 3)), 0.5)


# ---------------------------------------------------------------- Gaussian projection, refreshed seeds
def test_gaussian_normals_distribution():
    from scipy import stats

    from oracle import gaussian as og

    z = og.normals(2024, 3, 256, 4096)
    flat = z.ravel()
    n = flat.size
    # Kolmogorov–Smirnov against N(0, 1), for all draws and for the cosine and
    # sine outputs of the pairs separately
    assert stats.kstest(flat, "norm").pvalue > 1e-3
    assert stats.kstest(z[:, 0::4].ravel(), "norm").pvalue > 1e-3
    assert stats.kstest(z[:, 1::4].ravel(), "norm").pvalue > 1e-3
    # moments: mean 0, variance 1, skewness 0, kurtosis 3
    se = 1.0 / np.sqrt(n)
    assert abs(flat.mean()) < 5 * se
    assert abs(flat.var() - 1.0) < 5 * np.sqrt(2.0) * se
    assert abs(stats.skew(flat)) < 5 * np.sqrt(6.0) * se
    assert abs(stats.kurtosis(flat, fisher=False) - 3.0) < 5 * np.sqrt(24.0) * se
    # the two outputs of one pair, and neighbouring quads, are uncorrelated
    m = z[:, 0::4].size
    assert abs(np.corrcoef(z[:, 0::4].ravel(), z[:, 1::4].ravel())[0, 1]) < 5 / np.sqrt(m)
    assert abs(np.corrcoef(z[:, 0::4].ravel(), z[:, 2::4].ravel())[0, 1]) < 5 / np.sqrt(m)
    assert abs(np.corrcoef(z[:, :-4].ravel(), z[:, 4:].ravel())[0, 1]) < 5 / np.sqrt(z[:, 4:].size)
    # symmetric about zero
    assert abs((flat > 0).mean() - 0.5) < 5 * 0.5 * se


def test_gaussian_projection_structure():
    from oracle import gaussian as og
    from oracle import merge as omerge

    # a row depends only on (seed, stream, row): prefixes agree across sizes
    big = og.normals(9, 4, 12, 203)
    assert np.array_equal(og.normals(9, 4, 5, 37), big[:5, :37])
    assert not np.array_equal(og.normals(9, 5, 12, 203), big)      # stream id matters
    assert not np.array_equal(og.normals(10, 4, 12, 203), big)     # seed matters
    # the operand is the bf16 rounding of z and A = Ã/√r
    assert np.array_equal(og.operand(9, 4, 12, 203), omerge.bf16_round(big))
    assert np.allclose(og.projection(9, 4, 12, 203), omerge.bf16_round(big) / np.sqrt(12), rtol=0, atol=0)
    # E[AᵀA] = I over independent draws
    r, k, trials = 8, 6, 3000
    acc = np.zeros((k, k))
    for s in range(trials):
        A = og.projection(1000 + s, 0, r, k)
        acc += A.T @ A
    assert np.abs(acc / trials - np.eye(k)).max() < 0.06


def test_refreshed_seed_properties():
    seeds = [oph.refreshed_seed(105, t) for t in range(2000)]
    assert len(set(seeds)) == len(seeds)                    # a new key every step
    assert 105 not in seeds
    assert all(0 <= s < 2**64 for s in seeds)
    assert oph.refreshed_seed(105, 7) == oph.refreshed_seed(105, 7)
    assert oph.refreshed_seed(106, 7) != oph.refreshed_seed(105, 7)
    bits = np.array([bin(s).count("1") for s in seeds])
    assert abs(bits.mean() - 32.0) < 0.5                    # balanced bits
    # consecutive steps give unrelated projections
    a0 = oph.signs(seeds[0], 0, 16, 256).astype(np.float64)
    a1 = oph.signs(seeds[1], 0, 16, 256).astype(np.float64)
    assert abs((a0 * a1).mean()) < 5 / np.sqrt(a0.size)
    with pytest.raises(ValueError):
        oph.refreshed_seed(1, -1)


def test_gaussian_draws_independent_of_the_signs():
    # the Gaussian stream must not reuse the sign stream's generator calls: the
    # radius of a pair (a function of its first word) would then track the
    # number of −1 entries in the first 32 sign columns of the same call
    from oracle import gaussian as og

    xs, ys = [], []
    for seed in range(4):
        r, quads = 64, 64
        z = og.normals(500 + seed, 2, r, 4 * quads)
        b = oph.sign_bits(500 + seed, 2, r, 128 * quads)
        xs.append(b.reshape(r, quads, 128)[:, :, :32].sum(-1).ravel())
        ys.append((z[:, 0::4] ** 2 + z[:, 1::4] ** 2).ravel())
    c = np.corrcoef(np.concatenate(xs), np.concatenate(ys))[0, 1]
    assert abs(c) < 5 / np.sqrt(np.concatenate(xs).size)  # a shared call gives ≈ −0.32


# ---------------------------------------------------------------- reconstruction diagnostic
def test_reconstruction_cosine_pins():
    from oracle import diagnostic as odiag

    rng = np.random.default_rng(11)
    T, d, k, r = 40, 12, 30, 6
    # orthonormal rows whose span holds every row of G: exact reconstruction
    Q, _ = np.linalg.qr(rng.standard_normal((k, r)))
    A = Q.T                                              # r×k, AAᵀ = I
    X = rng.standard_normal((T, r)) @ A                  # rows of X in the row space of A
    dY = rng.standard_normal((T, d))
    assert abs(odiag.reconstruction_cosine(X, dY, A) - 1.0) < 1e-12
    # scale invariance in X and dY
    X2, dY2 = rng.standard_normal((T, k)), rng.standard_normal((T, d))
    As = oph.projection(3, 1, r, k)
    c = odiag.reconstruction_cosine(X2, dY2, As)
    assert abs(odiag.reconstruction_cosine(7.0 * X2, 1e-3 * dY2, As) - c) < 1e-12
    assert 0.0 < c < 1.0
    # the numerator is the squared norm of the sketch: cos·‖G‖·‖R‖ = ‖S‖²
    G = dY2.T @ X2
    S = G @ As.T
    assert abs(c * np.linalg.norm(G) * np.linalg.norm(S @ As) - np.sum(S * S)) < 1e-9 * np.sum(S * S)
    # random gradients: the value concentrates at tr(AAᵀ)/√(k‖AAᵀ‖²), close to √(r/(r+k)) for signs
    d_big, k_big, r_big = 400, 512, 32
    A = oph.projection(5, 0, r_big, k_big)
    G = rng.standard_normal((d_big, k_big))
    # G = dYᵀX with dY = I (T = d) and X = G reproduces a chosen dense gradient
    cval = odiag.reconstruction_cosine(G, np.eye(d_big), A)
    AA = A @ A.T
    expect = np.trace(AA) / np.sqrt(k_big * np.sum(AA * AA))
    assert abs(cval - expect) < 0.02
    assert abs(expect - np.sqrt(r_big / (r_big + k_big))) < 0.01


def test_merge_tolerance_helper_separates_cancellation():
    # The merge parity checker (tests/merge_tolerance.py) must reject an error
    # of two ulps on an ordinary weight, and accept a larger error only where
    # W − u cancels to a small fraction of its terms.  Planted here on the CPU.
    from merge_tolerance import check

    rng = np.random.default_rng(5)
    d, k, r, ae = 8, 32, 4, 1e-1
    A = oph.projection(3, 1, r, k)
    S = rng.standard_normal((d, r)) * 0.05
    W0 = omerge.bf16_round(rng.standard_normal((d, k)) * 0.02)
    u = ae * (S @ A)
    W0[2, 5] = omerge.bf16_round(u[2, 5])          # W ≈ u: the result cancels
    ref = omerge.merge(W0, S, A, ae)
    assert check(ref.copy(), ref, W0, S, A, ae) == 0
    got = ref.copy()
    got[1, 3] += 2 * omerge.bf16_ulp(ref[1, 3])     # two ulps on an ordinary weight
    with pytest.raises(AssertionError):
        check(got, ref, W0, S, A, ae)
    got = ref.copy()
    terms = ae * (np.abs(S) @ np.abs(A))
    extra = 2.0**-15 * terms[2, 5]                   # inside the allowance, beyond the ulp of a cancelled value
    assert extra > omerge.bf16_ulp(ref[2, 5])
    got[2, 5] += extra
    assert check(got, ref, W0, S, A, ae) == 1
