"""fp64 CPU oracle for the LoGRA low-rank gradient-sketching hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA path: the only module both sides use is
``synthetic.py``, which draws seeded inputs and holds none of the method's
arithmetic.

Source of every formula: "LoGRA: Scaling LLM Reinforcement Learning with
Low-Rank Gradient Sketches" (wispaper.ai summary page), sections
"草图如何取代完整梯度缓冲" (the sketch S = G Aᵀ, the projection A, the merge
W ← W − αηUA), "同一份草图也压缩策略同步开销" (A regenerated from a seed) and
"预测 KL 控制防止过大更新破坏学习" (predicted KL q(D) and
α = min{α_max, √(δ/q(D))}).

Modules
-------
philox   Philox4x32-10 written from Salmon et al., "Parallel random numbers:
         as easy as 1, 2, 3" (SC'11), plus the sign-to-projection mapping.
sketch   S = Σ_m (dY_mᵀ X_m) Aᵀ with the dense gradient formed explicitly.
merge    W′ = bf16_rne(W − αη·S·A) and an exact fp64→bf16 rounding.
kl       q(D) = mean over rows of KL(softmax(a/τ) ‖ softmax(b/τ)).
step     α = min(α_max, √(δ/q)) and the δ budget schedule.
momentum M ← β·M + S on the sketch (a reading; the pages give no rule).
gaussian Box–Muller normals from Philox and the bf16 Gaussian projection.
diagnostic cos(G, S·A), the gradient-reconstruction diagnostic.

Pinning status of each function is listed in the module headers; every
function is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle.py``.
"""

from . import philox, sketch, merge, kl, step, momentum, gaussian, diagnostic  # noqa: F401
