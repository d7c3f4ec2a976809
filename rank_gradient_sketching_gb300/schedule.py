"""KL budget schedule for the step-size controller.

LoGRA summary page, section "预测 KL 控制防止过大更新破坏学习": the budget δ is
constant or annealed so that later training allows smaller policy changes;
section "这些节省能说明什么、不能说明什么" anneals it from 2×10⁻⁴ to 2×10⁻⁵.
The pages give only the endpoints; this schedule interpolates linearly, with
both endpoints included.
"""

from __future__ import annotations


def delta_schedule(delta_start: float, delta_end: float, steps: int) -> list[float]:
    if steps < 1:
        raise ValueError("steps must be >= 1")
    if steps == 1:
        return [float(delta_start)]
    span = float(delta_end) - float(delta_start)
    return [float(delta_start) + span * (i / (steps - 1)) for i in range(steps)]
