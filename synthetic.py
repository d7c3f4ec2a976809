"""Seeded synthetic inputs for the LoGRA sketching hot path.

This module only draws random numbers of the workloads' shapes and
distributions; it holds none of the method's arithmetic (no projection, no
sketch, no merge, no KL).  Both the CUDA path's tests/bench and the oracle take
their inputs from here, so it must stay free of either side's code.

Workloads (all synthetic; the pages' own runs used Qwen2.5-Math-1.5B / 7B on
DAPO-Math-7.5k and MATH-500, none of which is available here — these shapes and
distributions stand in for them):

tiny      one 256×256 layer, r=4, 2 micro-batches of 128 tokens, X ~ N(0,1),
          dY ~ N(0,1e-3), W ~ N(0,0.02), projection seed 0, αη = 1e-3;
          predicted KL on 16 rows × vocab 1024, fp32 logits ~ N(0,2),
          proposed = current + 0.05·N(0,1), τ = 1, δ = 2e-4, α_max = 1.
square    d = k = 4096, r = 64, 8 micro-batches of 4096 tokens, dY ~ N(0,1e-4),
          projection seed 1, one merge with αη = 2e-4.
qwen1.5b  hidden 1536, 28 layers, q/o 1536×1536, k/v 256×1536, gate/up
          8960×1536, down 1536×8960; r ∈ {4,16,64,256}; micro-batch 8×1024 =
          8192 tokens; 4 micro-batches; per-layer seed 100+layer.
qwen7b    hidden 3584, 28 layers, q/o 3584×3584, k/v 512×3584, gate/up
          18944×3584, down 3584×18944; r ∈ {256, 64}; micro-batch 16×1024 =
          16384 tokens; 8 micro-batches then one merge with αη = 2e-4.
kl        64 responses × 1024 tokens = 65536 rows × vocab 151936, bf16 current
          logits ~ N(0,3) with ⌊V/100⌋ distinct entries per row boosted by +8,
          proposed = current + ε·N(0,1) (fp32, then stored as bf16), ε ∈ {0.01,
          0.1}, τ = 1, δ annealed 2e-4 → 2e-5 over 10 steps, α_max = 1.

N(μ, σ) is read with σ a standard deviation.  Every tensor has its own seed,
derived from (workload, layer, matrix, micro-batch, tensor name).
"""

from __future__ import annotations

import zlib

import torch

# (name, stream_id) of the seven sketched projections of one decoder layer, in
# the order q, k, v, o, gate, up, down.
PROJECTIONS = ("q", "k", "v", "o", "gate", "up", "down")


def layer_shapes(hidden: int, kv: int, ffn: int) -> list[tuple[str, int, int, int]]:
    """[(name, d, k, stream_id)] for one decoder layer (W is d×k, out×in)."""
    return [
        ("q", hidden, hidden, 0),
        ("k", kv, hidden, 1),
        ("v", kv, hidden, 2),
        ("o", hidden, hidden, 3),
        ("gate", ffn, hidden, 4),
        ("up", ffn, hidden, 5),
        ("down", hidden, ffn, 6),
    ]


WORKLOADS = {
    "tiny": dict(layers=[[("w", 256, 256, 0)]], r=(4,), tokens=128, microbatches=2,
                 x_std=1.0, dy_std=1e-3, w_std=0.02, seeds=[0], alpha_eta=1e-3),
    "square": dict(layers=[[("w", 4096, 4096, 0)]], r=(64,), tokens=4096, microbatches=8,
                   x_std=1.0, dy_std=1e-4, w_std=0.02, seeds=[1], alpha_eta=2e-4),
    "qwen1.5b": dict(layers=[layer_shapes(1536, 256, 8960)] * 28, r=(4, 16, 64, 256), tokens=8192,
                     microbatches=4, x_std=1.0, dy_std=1e-4, w_std=0.02,
                     seeds=[100 + i for i in range(28)], alpha_eta=2e-4),
    "qwen7b": dict(layers=[layer_shapes(3584, 512, 18944)] * 28, r=(256, 64), tokens=16384,
                   microbatches=8, x_std=1.0, dy_std=1e-4, w_std=0.02,
                   seeds=[100 + i for i in range(28)], alpha_eta=2e-4),
}

KL_WORKLOADS = {
    "tiny": dict(rows=16, vocab=1024, std=2.0, eps=(0.05,), boost_frac=0.0, boost=0.0,
                 dtype=torch.float32, temperature=1.0, delta=(2e-4, 2e-4), steps=1, alpha_max=1.0),
    "qwen": dict(rows=64 * 1024, vocab=151936, std=3.0, eps=(0.01, 0.1), boost_frac=0.01, boost=8.0,
                 dtype=torch.bfloat16, temperature=1.0, delta=(2e-4, 2e-5), steps=10, alpha_max=1.0),
}


def seed_of(*parts) -> int:
    """A stable 63-bit seed from a tuple of labels."""
    h = zlib.crc32(repr(parts).encode())
    h2 = zlib.crc32(repr(parts[::-1]).encode())
    return ((h << 31) ^ h2) & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, device="cpu", dtype=torch.bfloat16,
           chunk_elems: int = 1 << 28) -> torch.Tensor:
    """std·N(0,1) drawn in fp32 and stored as `dtype`, generated in row chunks
    so that large tensors need no full-size fp32 temporary."""
    out = torch.empty(shape, dtype=dtype, device=device)
    g = _gen(seed, device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        tmp = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:e].copy_(tmp)
    return out


def microbatch(workload: str, layer: int, name: str, mb: int, T: int, d: int, k: int, device="cpu"):
    """(X T×k bf16, dY T×d bf16) of one micro-batch for one matrix."""
    w = WORKLOADS[workload]
    X = normal((T, k), w["x_std"], seed_of(workload, layer, name, mb, "X"), device)
    dY = normal((T, d), w["dy_std"], seed_of(workload, layer, name, mb, "dY"), device)
    return X, dY


def weight(workload: str, layer: int, name: str, d: int, k: int, device="cpu") -> torch.Tensor:
    w = WORKLOADS[workload]
    return normal((d, k), w["w_std"], seed_of(workload, layer, name, "W"), device)


def kl_logits(workload: str, eps: float, rows: int | None = None, vocab: int | None = None,
              device="cpu", row_chunk: int = 1024):
    """(current, proposed) logits, rows × vocab, in the workload's dtype.

    current = std·N(0,1) with ⌊vocab·boost_frac⌋ distinct uniformly chosen
    entries per row raised by `boost`; proposed = current + eps·N(0,1),
    computed in fp32 and then stored in the workload's dtype.
    """
    w = KL_WORKLOADS[workload]
    rows = w["rows"] if rows is None else rows
    vocab = w["vocab"] if vocab is None else vocab
    dtype = w["dtype"]
    cur = torch.empty((rows, vocab), dtype=dtype, device=device)
    prop = torch.empty((rows, vocab), dtype=dtype, device=device)
    g_cur = _gen(seed_of(workload, "cur", rows, vocab), device)
    g_sel = _gen(seed_of(workload, "boost", rows, vocab), device)
    g_eps = _gen(seed_of(workload, "prop", eps, rows, vocab), device)
    nboost = int(vocab * w["boost_frac"])
    for s in range(0, rows, row_chunk):
        e = min(rows, s + row_chunk)
        a = torch.randn((e - s, vocab), generator=g_cur, device=device, dtype=torch.float32)
        a.mul_(w["std"])
        if nboost:
            keys = torch.rand((e - s, vocab), generator=g_sel, device=device, dtype=torch.float32)
            idx = torch.topk(keys, nboost, dim=1).indices
            a.scatter_add_(1, idx, torch.full(idx.shape, w["boost"], device=device, dtype=torch.float32))
        a_st = a.to(dtype)
        cur[s:e].copy_(a_st)
        noise = torch.randn((e - s, vocab), generator=g_eps, device=device, dtype=torch.float32)
        prop[s:e].copy_(a_st.float() + eps * noise)
    return cur, prop
