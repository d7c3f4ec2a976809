"""Step-size controller α = min(α_max, √(δ/q(D))) and the δ budget (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LoGRA summary page, section "预测 KL 控制防止过大更新破坏学习": the mean
predicted KL scales as α²·q(D); for a KL budget δ the controller sets
α = min{α_max, √(δ/q(D))}, so q(D) = 4δ gives α = 1/2 and α_max stops small
q(D) from blowing the step up.  The budget is constant or annealed
(decreasing); the LoRA comparison in section "这些节省能说明什么、不能说明什么"
anneals it from 2×10⁻⁴ to 2×10⁻⁵.

Readings: q(D) = 0 (or a negative rounding residue) gives α = α_max; NaN q
gives NaN; the anneal is linear over the given number of steps, endpoints
included (the pages give only the endpoints).

Pinned by: q = 4δ ⇒ α = 1/2, the α_max cap, the q = 0 case, and the
α²-scaling of the predicted KL (tests/test_oracle.py).
"""

from __future__ import annotations

import math

import numpy as np


def step_size(q: float, delta: float, alpha_max: float) -> float:
    if not (delta > 0 and alpha_max > 0):
        raise ValueError("delta and alpha_max must be > 0")
    if math.isnan(q):
        return math.nan
    if q <= 0:
        return float(alpha_max)
    return float(min(alpha_max, math.sqrt(delta / q)))


def delta_schedule(delta_start: float, delta_end: float, steps: int) -> np.ndarray:
    """Linearly annealed budget, `steps` values from delta_start to delta_end."""
    if steps < 1:
        raise ValueError("steps must be >= 1")
    if steps == 1:
        return np.array([float(delta_start)])
    return np.array([delta_start + (delta_end - delta_start) * i / (steps - 1) for i in range(steps)])
