"""The merge tolerance, and where its cancellation allowance applies.

The merged weight W' = bf16_rn(W − αη·S·A) is checked against the oracle's
value rounded to bf16.  The bound is one bf16 ulp of that value, plus a
dot-product error term 2⁻¹⁴·|αη|·(|S|·|A|) (Higham's γ·Σ|x||y| form at 2⁻¹⁴
relative) for results that cancel: where W − u is far smaller than the terms
that form it, any fp32 evaluation of u moves the result by more than the ulp
of the cancelled value.

`check` asserts the bound everywhere, and also that every weight outside a
strict 1-ulp bound is such a cancellation (|W'| ≤ 2⁻⁸ of |W| + |αη|·(|S|·|A|)).
It returns the number of weights that needed the allowance, which the
workload tests print and bound.
"""

import numpy as np

import oracle.merge as omerge


def check(got, ref, W0, S, A, alpha_eta, what="merge"):
    got, ref, W0 = (np.asarray(x, dtype=np.float64) for x in (got, ref, W0))
    terms = abs(alpha_eta) * (np.abs(np.asarray(S, dtype=np.float64)) @ np.abs(np.asarray(A, dtype=np.float64)))
    ulp = omerge.bf16_ulp(ref)
    err = np.abs(got - ref)
    bound = ulp + 2.0**-14 * terms
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} weights outside the bound; worst {err[bad].max()}"
    strict = err > ulp
    cancelled = np.abs(ref) <= 2.0**-8 * (np.abs(W0) + terms)
    odd = strict & ~cancelled
    assert not odd.any(), (f"{what}: {odd.sum()} weights outside 1 bf16 ulp without cancellation "
                           f"(e.g. got {got[odd][0]}, want {ref[odd][0]}, W {W0[odd][0]})")
    return int(strict.sum())
