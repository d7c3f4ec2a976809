"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching the device."""

import ctypes
import math
import os
import re

import pytest

from oracle import philox as oph

from oracle import step as ostep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lg():
    import __graft_entry__

    __graft_entry__.build()
    import rank_gradient_sketching_gb300 as mod

    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "logra.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(logra_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_path(lg):
    names = _declared()
    for n in ["logra_sketch_accumulate", "logra_merge_update", "logra_regen_projection", "logra_predicted_kl",
              "logra_step_size"]:
        assert n in names


def test_every_declared_symbol_is_exported(lg):
    for name in _declared():
        assert hasattr(lg.lib, name), name  # ctypes resolves through dlsym


def test_version_and_status_strings(lg):
    assert lg.logra_version() >= 100
    assert lg.lib.logra_status_string(0) == b"LOGRA_OK"
    assert lg.lib.logra_status_string(4) == b"LOGRA_ERR_WORKSPACE"


def _sketch(lg, **kw):
    a = dict(X=16, ldx=256, dY=16, lddy=256, T=128, d=256, k=256, r=4, seed=0, sid=0, S=16, lds=4, ws=256,
             wsb=1 << 30, stream=None)
    a.update(kw)
    return lg.lib.logra_sketch_accumulate(a["X"], a["ldx"], a["dY"], a["lddy"], a["T"], a["d"], a["k"], a["r"],
                                          a["seed"], a["sid"], a["S"], a["lds"], a["ws"], a["wsb"], a["stream"])


def test_sketch_validation_on_host(lg):
    assert _sketch(lg, r=0) == 1
    assert _sketch(lg, r=257) == 5
    assert _sketch(lg, T=-1) == 2
    assert _sketch(lg, X=None) == 1
    assert _sketch(lg, ldx=100) == 2
    assert _sketch(lg, lds=2) == 2
    assert _sketch(lg, X=8) == 3        # not 16-byte aligned
    assert _sketch(lg, ldx=260) == 3    # not a multiple of 8
    assert _sketch(lg, ws=128) == 3     # workspace not 256-byte aligned
    assert _sketch(lg, d=130) == 3      # row of dY not a whole number of 16-byte units
    assert _sketch(lg, k=250) == 3
    assert _sketch(lg, wsb=16) == 4
    assert "workspace" in lg.logra_last_error()
    # empty problems are no-ops and touch nothing
    assert _sketch(lg, T=0, X=None, dY=None, S=None, ws=None) == 0
    assert lg.logra_last_error() == ""


def test_sketch_workspace_formula(lg):
    T, d, k, r = 1000, 300, 500, 20
    np16, Tp, dp = 32, 1024, 384
    al = lambda x: (x + 255) // 256 * 256
    # above r = 64, P is fp16 in blocks of 64 tokens, each two halves of 64
    # fp32 token scales + 56 rows × 128 bytes, and rows are padded to CTA pairs (256)
    s100 = lg.logra_sketch_splits(T, d, k, 100)
    assert lg.logra_sketch_workspace_bytes(T, d, k, 100) == al((Tp // 64) * 2 * (256 + 112 * 64)) + (
        al(s100 * 512 * 112 * 4) if s100 > 1 else 0)
    splits = lg.logra_sketch_splits(T, d, k, r)
    assert splits >= 1
    al = lambda x: (x + 255) // 256 * 256
    want = 2 * al(np16 * Tp * 2) + (al(splits * dp * np16 * 4) if splits > 1 else 0)
    assert lg.logra_sketch_workspace_bytes(T, d, k, r) == want
    # the split count depends on the shape only and partitions T
    assert lg.logra_sketch_splits(16384, 3584, 3584, 64) == lg.logra_sketch_splits(16384, 3584, 3584, 64)
    assert lg.logra_sketch_workspace_bytes(-1, 1, 1, 1) == 0


def test_merge_validation_on_host(lg):
    f = lg.lib.logra_merge_update
    assert f(16, 256, 256, 256, 16, 4, 0, 0, 0, 1e-3, None, None) == 1           # r = 0
    assert f(16, 256, 256, 256, 16, 4, 300, 0, 0, 1e-3, None, None) == 5         # r > 256
    assert f(16, 256, 256, 256, 16, 4, 4, 0, 0, math.nan, None, None) == 1       # non-finite αη
    assert f(None, 256, 256, 256, 16, 4, 4, 0, 0, 1e-3, None, None) == 1
    assert f(16, 100, 256, 256, 16, 4, 4, 0, 0, 1e-3, None, None) == 2
    assert f(8, 256, 256, 256, 16, 4, 4, 0, 0, 1e-3, None, None) == 3
    assert f(16, 256, 256, 250, 16, 4, 4, 0, 0, 1e-3, None, None) == 3           # k not a multiple of 8
    assert f(16, 256, 0, 256, None, 4, 4, 0, 0, 1e-3, None, None) == 0           # d = 0: no-op


def test_momentum_validation_on_host(lg):
    f = lg.lib.logra_sketch_momentum
    assert f(16, 64, 32, 64, 8, 0, 0.9, 0, None) == 1              # r = 0
    assert f(16, 512, 32, 512, 8, 300, 0.9, 0, None) == 5          # r > 256
    assert f(16, 64, 32, 64, -1, 64, 0.9, 0, None) == 2            # d < 0
    assert f(16, 64, 32, 64, 8, 64, math.inf, 0, None) == 1        # non-finite β
    assert f(None, 64, 32, 64, 8, 64, 0.9, 0, None) == 1
    assert f(16, 64, 16, 64, 8, 64, 0.9, 0, None) == 1             # M == S
    assert f(16, 32, 32, 64, 8, 64, 0.9, 0, None) == 2             # ldm < r
    assert f(16, 64, 32, 63, 8, 64, 0.9, 0, None) == 2             # lds < r
    assert f(18, 64, 32, 64, 8, 64, 0.9, 0, None) == 3             # M not 4-byte aligned
    assert f(None, 64, None, 64, 0, 64, 0.9, 1, None) == 0         # d = 0: no-op


def test_explicit_projection_validation_on_host(lg):
    f = lg.lib.logra_sketch_accumulate_proj
    ok = dict(X=16, ldx=256, dY=16, lddy=256, T=128, d=256, k=256, r=4, A=16, lda=256, S=16, lds=4, ws=256,
              wsb=1 << 30, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*a.values())

    assert call(A=None) == 1                       # no operand
    assert call(lda=200) == 2                      # lda < k
    assert call(A=24) == 3                         # operand not 16-byte aligned
    assert call(lda=260) == 3                      # lda not a multiple of 8
    assert call(r=0) == 1 and call(r=257) == 5     # same rank checks as the sign path
    assert call(T=0, A=None) == 0                  # empty: no-op before the operand is looked at
    m = lg.lib.logra_merge_update_proj
    assert m(16, 256, 256, 256, 16, 4, 4, None, 256, 1e-3, None, None) == 1
    assert m(16, 256, 256, 256, 16, 4, 4, 16, 100, 1e-3, None, None) == 2
    assert m(16, 256, 256, 256, 16, 4, 4, 8, 256, 1e-3, None, None) == 3
    assert m(16, 256, 256, 256, 16, 4, 4, 16, 256, math.nan, None, None) == 1
    assert m(16, 256, 0, 256, None, 4, 4, None, 256, 1e-3, None, None) == 0
    g = lg.lib.logra_regen_projection
    assert g(1, 0, 4, 256, 9, 16, 256, None) == 5          # unknown kind
    assert g(1, 0, 4, 256, lg.LOGRA_PROJ_GAUSS_FP32, 18, 256, None) == 3  # fp32 output not 4-byte aligned


def test_sum_squares_validation_on_host(lg):
    f = lg.lib.logra_sum_squares
    wsb = lg.lib.logra_sum_squares_workspace_bytes()
    assert wsb >= 8
    assert f(16, 7, 4, 4, 4, 16, 0, 256, wsb, None) == 5           # unknown dtype
    assert f(16, 1, -1, 4, 4, 16, 0, 256, wsb, None) == 2          # negative rows
    assert f(16, 1, 4, 4, 4, None, 0, 256, wsb, None) == 1         # no output
    assert f(16, 1, 4, 4, 4, 12, 0, 256, wsb, None) == 3           # output not 8-byte aligned
    assert f(None, 1, 4, 4, 4, 16, 0, 256, wsb, None) == 1         # no input
    assert f(16, 1, 4, 8, 4, 16, 0, 256, wsb, None) == 2           # ld < cols
    assert f(18, 1, 4, 4, 4, 16, 0, 256, wsb, None) == 3           # fp32 input not 4-byte aligned
    assert f(16, 1, 4, 4, 4, 16, 0, 256, wsb - 8, None) == 4       # workspace too small


def test_shared_x_proj_validation_on_host(lg):
    import ctypes

    from rank_gradient_sketching_gb300._binding import logra_sketch_target

    f = lg.lib.logra_sketch_accumulate_shared_x_proj
    tg = (logra_sketch_target * 1)()
    tg[0] = logra_sketch_target(16, 256, 256, 0, 0, 16, 4)
    ops = (ctypes.c_void_p * 1)(16)
    ldas = (ctypes.c_int64 * 1)(256)
    assert f(16, 256, 128, 256, 1, tg, None, ldas, 4, 256, 1 << 30, None) == 1   # no operands
    bad = (ctypes.c_void_p * 1)(24)
    assert f(16, 256, 128, 256, 1, tg, bad, ldas, 4, 256, 1 << 30, None) == 3    # operand not 16-byte aligned
    short = (ctypes.c_int64 * 1)(100)
    assert f(16, 256, 128, 256, 1, tg, ops, short, 4, 256, 1 << 30, None) == 2   # lda < k
    assert f(16, 256, 0, 256, 1, tg, ops, ldas, 4, 256, 1 << 30, None) == 0      # T = 0: no-op


def test_refreshed_seed_matches_oracle(lg):
    # a host function: the library's value against the oracle's definition
    for base, step in [(105, 0), (105, 1), (0, 0), (2**64 - 1, 2**40 + 3), (123456789, 987654321)]:
        assert lg.logra_refreshed_seed(base, step) == oph.refreshed_seed(base, step)


def test_kl_validation_on_host(lg):
    f = lg.lib.logra_predicted_kl
    args = [16, 16, 0, 4, 1024, 1024, 1.0, None, 16, None, 256, 1 << 20, None]
    assert f(*args[:2], 7, *args[3:]) == 5                    # unknown dtype
    bad = list(args); bad[6] = 0.0
    assert f(*bad) == 1                                       # temperature 0
    bad = list(args); bad[6] = math.inf
    assert f(*bad) == 1
    bad = list(args); bad[4] = 0
    assert f(*bad) == 2                                       # V = 0
    bad = list(args); bad[5] = 1000
    assert f(*bad) == 2                                       # ld < V
    bad = list(args); bad[5] = 1028
    assert f(*bad) == 3                                       # ld not a multiple of 8 bf16
    bad = list(args); bad[11] = 8
    assert f(*bad) == 4                                       # workspace too small
    assert lg.logra_kl_workspace_bytes(1000) == 8192


def test_regen_validation_on_host(lg):
    f = lg.lib.logra_regen_projection
    assert f(0, 0, 4, 100, 9, 16, 100, None) == 5
    assert f(0, 0, 0, 100, 0, 16, 100, None) == 1
    assert f(0, 0, 4, 100, 0, None, 100, None) == 1
    assert f(0, 0, 4, 100, 0, 16, 50, None) == 2
    assert f(0, 0, 4, 0, 0, None, 0, None) == 0


@pytest.mark.parametrize("q", [0.0, -1e-9, 1e-6, 8e-4, 1.0, math.inf])
def test_host_step_size_matches_oracle(lg, q):
    for delta, amax in [(2e-4, 1.0), (2e-5, 0.3)]:
        assert lg.logra_step_size(q, delta, amax) == ostep.step_size(q, delta, amax)


def test_host_step_size_edges(lg):
    assert lg.logra_step_size(4 * 2e-4, 2e-4, 1.0) == 0.5
    assert math.isnan(lg.logra_step_size(math.nan, 2e-4, 1.0))
    with pytest.raises(lg.LograError):
        lg.logra_step_size(1.0, 0.0, 1.0)
    with pytest.raises(lg.LograError):
        lg.logra_step_size(1.0, 1e-4, -1.0)
    out = ctypes.c_double()
    assert lg.lib.logra_step_size(1.0, 1e-4, 1.0, None) == 1
    assert lg.lib.logra_step_size(1.0, 1e-4, 1.0, ctypes.byref(out)) == 0


def test_delta_schedule_matches_oracle(lg):
    a = lg.delta_schedule(2e-4, 2e-5, 10)
    b = ostep.delta_schedule(2e-4, 2e-5, 10)
    assert len(a) == 10 and all(math.isclose(x, y, rel_tol=1e-15) for x, y in zip(a, b))


def _aligned_buffer(nbytes, align=128):
    buf = ctypes.create_string_buffer(nbytes + align)
    addr = ctypes.addressof(buf)
    return buf, addr + (-addr) % align


def _merge_targets(lg, shapes, with_a=False):
    T = lg._binding.logra_merge_target
    arr = (T * max(1, len(shapes)))()
    for j, (d, k) in enumerate(shapes):
        arr[j] = T(4096 * (j + 1), k, d, k, 4096 * (j + 1) + 2048, 8, 7 + j, j, 4096 if with_a else None, k)
    return arr


def test_merge_group_plan_on_host(lg):
    # a plan whose weights are all empty (d or k = 0) needs no tensor maps and
    # is built here: a valid plan with nothing to launch
    import struct

    shapes = [(0, 64), (256, 0), (0, 0)]
    n, r = len(shapes), 64
    nbytes = lg.lib.logra_merge_group_plan_bytes(n)
    assert nbytes == 128 + 128 + 512 * n        # header, CTA offsets (rounded to 128 bytes), entries
    buf, plan = _aligned_buffer(nbytes)
    assert lg.lib.logra_merge_group_plan(n, _merge_targets(lg, shapes), r, plan, nbytes) == 0
    raw = ctypes.string_at(plan, nbytes)
    magic, n_, r_, np_, path, total = struct.unpack_from("<Iiiiii", raw, 0)
    assert (magic, n_, r_, np_, path, total) == (0x4C474D50, n, r, 64, 1, 0)
    assert struct.unpack_from(f"<{n + 1}i", raw, 128) == (0,) * (n + 1)
    assert lg.lib.logra_merge_group_plan(0, None, 4, plan, nbytes) == 0
    assert struct.unpack_from("<iiii", ctypes.string_at(plan, 24), 8) == (4, 16, 1, 0)  # r, np, path, CTAs


def test_merge_group_plan_ring_sizes_on_host(lg):
    # The ±1 ring a plan records: three tiles, two from np = 80 to 128 (two
    # CTAs per SM), and two above np = 128 with a given operand. There two
    # warps issue the MMAs of alternate chunks and tell a stage's phases apart
    # by parity; the operand tiles arrive by TMA, possibly out of order, so
    # each stage must belong to one issuer (an even ring).
    import struct

    shapes = [(0, 64), (256, 0)]
    n = len(shapes)
    nbytes = lg.lib.logra_merge_group_plan_bytes(n)
    buf, plan = _aligned_buffer(nbytes)
    cases = [(16, False, 3), (64, False, 3), (100, False, 2), (128, True, 2), (200, False, 3),
             (256, False, 3), (200, True, 2), (256, True, 2)]
    for r, with_a, want in cases:
        assert lg.lib.logra_merge_group_plan(n, _merge_targets(lg, shapes, with_a=with_a), r, plan, nbytes) == 0
        raw = ctypes.string_at(plan, 48)
        b_stages = struct.unpack_from("<i", raw, 28)[0]
        explicit_a = struct.unpack_from("<i", raw, 44)[0]
        assert (b_stages, explicit_a) == (want, int(with_a)), (r, with_a)


def test_merge_group_validation_on_host(lg):
    f = lg.lib.logra_merge_group_plan
    shapes = [(256, 256), (128, 512)]
    nbytes = lg.lib.logra_merge_group_plan_bytes(2)
    buf, plan = _aligned_buffer(nbytes)
    tg = _merge_targets(lg, shapes)
    assert f(-1, tg, 4, plan, nbytes) == 1                   # n < 0
    assert f(2, None, 4, plan, nbytes) == 1                  # no targets
    assert f(2, tg, 0, plan, nbytes) == 1                    # r = 0
    assert f(2, tg, 257, plan, nbytes) == 5                  # r > 256
    assert f(2, tg, 4, None, nbytes) == 1                    # no plan
    assert f(2, tg, 4, plan + 8, nbytes) == 3                # plan not 128-byte aligned
    assert f(2, tg, 4, plan, nbytes - 1) == 4                # plan too small
    mixed = _merge_targets(lg, shapes)
    mixed[1].A = 4096
    assert f(2, mixed, 4, plan, nbytes) == 1                 # operand on some targets only
    assert b"target 1" in lg.lib.logra_last_error()
    bad = _merge_targets(lg, shapes)
    bad[1].ldw = 100
    assert f(2, bad, 4, plan, nbytes) == 2                   # ldw < k on target 1
    bad = _merge_targets(lg, shapes)
    bad[0].k = 250
    bad[0].ldw = 256
    assert f(2, bad, 4, plan, nbytes) == 3                   # k not a multiple of 8
    bad = _merge_targets(lg, shapes)
    bad[1].W = 4104
    assert f(2, bad, 4, plan, nbytes) == 3                   # W not 16-byte aligned
    ops = _merge_targets(lg, shapes, with_a=True)
    ops[0].lda = 100
    assert f(2, ops, 4, plan, nbytes) == 2                   # operand row stride below k
    # W regions that share bytes (a weight named twice, tied weights) would
    # race inside one launch: refused before any plan is written
    over = _merge_targets(lg, shapes)                        # W at 4096 (256 rows of 512 B) and at 8192
    assert f(2, over, 4, plan, nbytes) == 1
    assert b"overlap" in lg.lib.logra_last_error()
    same = _merge_targets(lg, [(128, 64), (128, 64)])
    same[1].W = same[0].W                                    # one weight given twice
    assert f(2, same, 4, plan, nbytes) == 1
    u = lg.lib.logra_merge_update_group
    assert f(2, _merge_targets(lg, [(0, 64), (128, 0)]), 4, plan, nbytes) == 0   # a plan (no maps needed)
    assert u(None, plan, 1e-3, None, None) == 1              # no host plan
    assert u(plan, plan + 64, 1e-3, None, None) == 3         # device copy misaligned
    assert u(plan, plan, math.nan, None, None) == 1          # non-finite αη
    zeros, zp = _aligned_buffer(nbytes)
    assert u(zp, zp, 1e-3, None, None) == 1                  # not a plan


def _sketch_group_targets(lg, shapes, r=4, with_a=False):
    """Targets at fake, well-aligned addresses: X at 1 MiB·(j+1), dY half a
    MiB further, S at 64 MiB + 1 MiB·j (none overlap)."""
    T = lg._binding.logra_sketch_group_target
    arr = (T * max(1, len(shapes)))()
    for j, (t, d, k) in enumerate(shapes):
        x = (1 << 20) * (j + 1)
        arr[j] = T(x, k, x + (1 << 19), d, t, d, k, 7 + j, j, (1 << 30) if with_a else None, k,
                   (1 << 26) + (1 << 20) * j, r)
    return arr


def _group_plan_bytes(n, entry):
    a = lambda c: (4 * c + 127) // 128 * 128  # noqa: E731
    return 128 + 3 * (a(n + 1) + a(n)) + n * entry


def test_sketch_group_plan_on_host(lg):
    # a plan whose targets are all empty (T, d or k = 0) needs no tensor maps
    # and is built here: a valid plan with nothing to launch
    import struct

    shapes = [(0, 64, 64), (128, 0, 64), (128, 64, 0)]
    n, r = len(shapes), 100
    nbytes = lg.lib.logra_sketch_group_plan_bytes(n)
    entry = (nbytes - _group_plan_bytes(n, 0)) // n
    assert entry % 128 == 0 and nbytes == _group_plan_bytes(n, entry)
    assert lg.lib.logra_sketch_group_plan_bytes(n + 40) == _group_plan_bytes(n + 40, entry)
    tg = _sketch_group_targets(lg, shapes, r)
    assert lg.lib.logra_sketch_group_workspace_bytes(n, tg, r) == 0
    buf, plan = _aligned_buffer(nbytes)
    assert lg.lib.logra_sketch_group_plan(n, tg, r, None, 0, plan, nbytes) == 0  # no workspace needed
    raw = ctypes.string_at(plan, nbytes)
    magic, n_, r_, np_, p16, proj, con, red = struct.unpack_from("<Iiiiiiii", raw, 0)
    assert (magic, n_, r_, np_, p16, proj, con, red) == (0x4C475350, n, r, 112, 1, 0, 0, 0)
    for phase in range(3):  # every matrix of every phase starts at CTA 0 (none has any)
        off = 128 + phase * ((4 * (n + 1) + 127) // 128 * 128 + (4 * n + 127) // 128 * 128)
        assert struct.unpack_from(f"<{n + 1}i", raw, off) == (0,) * (n + 1)
    assert lg.lib.logra_sketch_group_plan(0, None, 4, None, 0, plan, nbytes) == 0


def test_sketch_group_workspace_formula(lg):
    # target j's region is laid out as for one call, each rounded up to 256
    # bytes; an empty target (T, d or k = 0) takes none
    shapes = [(1000, 304, 520), (0, 64, 64), (4096, 256, 512), (77, 64, 64)]
    for r in (4, 64, 100, 256):
        tg = _sketch_group_targets(lg, shapes, r)
        want = sum((lg.logra_sketch_workspace_bytes(t, d, k, r) + 255) // 256 * 256 for (t, d, k) in shapes
                   if t and d and k)
        assert lg.lib.logra_sketch_group_workspace_bytes(len(shapes), tg, r) == want
    assert lg.lib.logra_sketch_group_workspace_bytes(-1, tg, 4) == 0
    assert lg.lib.logra_sketch_group_workspace_bytes(2, tg, 0) == 0
    assert lg.lib.logra_sketch_group_workspace_bytes(2, tg, 257) == 0
    bad = _sketch_group_targets(lg, [(-1, 8, 8)], 4)
    assert lg.lib.logra_sketch_group_workspace_bytes(1, bad, 4) == 0


def test_sketch_group_validation_on_host(lg):
    f = lg.lib.logra_sketch_group_plan
    shapes = [(256, 256, 256), (128, 128, 512)]
    r = 4
    nbytes = lg.lib.logra_sketch_group_plan_bytes(2)
    buf, plan = _aligned_buffer(nbytes)
    ws, wsb = 1 << 32, 1 << 40                                    # a fake, aligned workspace
    tg = _sketch_group_targets(lg, shapes, r)
    assert f(-1, tg, r, ws, wsb, plan, nbytes) == 1              # n < 0
    assert f(2, None, r, ws, wsb, plan, nbytes) == 1             # no targets
    assert f(2, tg, 0, ws, wsb, plan, nbytes) == 1               # r = 0
    assert f(2, tg, 257, ws, wsb, plan, nbytes) == 5             # r > 256
    assert f(2, tg, r, ws, wsb, None, nbytes) == 1               # no plan
    assert f(2, tg, r, ws, wsb, plan + 8, nbytes) == 3           # plan not 128-byte aligned
    assert f(2, tg, r, ws, wsb, plan, nbytes - 1) == 4           # plan too small
    assert f(2, tg, r, None, wsb, plan, nbytes) == 1             # no workspace
    assert f(2, tg, r, ws + 128, wsb, plan, nbytes) == 3         # workspace not 256-byte aligned
    need = lg.lib.logra_sketch_group_workspace_bytes(2, tg, r)
    assert f(2, tg, r, ws, need - 1, plan, nbytes) == 4          # workspace too small
    bad = _sketch_group_targets(lg, shapes, r)
    bad[1].ldx = 100
    assert f(2, bad, r, ws, wsb, plan, nbytes) == 2              # ldx < k on target 1
    assert b"target 1" in lg.lib.logra_last_error()
    bad = _sketch_group_targets(lg, shapes, r)
    bad[0].lds = 2
    assert f(2, bad, r, ws, wsb, plan, nbytes) == 2              # lds < r
    bad = _sketch_group_targets(lg, shapes, r)
    bad[0].d = 250
    bad[0].lddy = 256
    assert f(2, bad, r, ws, wsb, plan, nbytes) == 3              # d not a multiple of 8
    bad = _sketch_group_targets(lg, shapes, r)
    bad[1].dY = bad[1].dY + 8
    assert f(2, bad, r, ws, wsb, plan, nbytes) == 3              # dY not 16-byte aligned
    bad = _sketch_group_targets(lg, shapes, r)
    bad[1].X = None
    assert f(2, bad, r, ws, wsb, plan, nbytes) == 1              # X missing
    ops = _sketch_group_targets(lg, shapes, r, with_a=True)
    ops[0].lda = 100
    assert f(2, ops, r, ws, wsb, plan, nbytes) == 2              # operand row stride below k
    # S regions that share bytes would race inside one launch: refused
    # before any plan is written
    same = _sketch_group_targets(lg, shapes, r)
    same[1].S = same[0].S                                        # one sketch given twice
    assert f(2, same, r, ws, wsb, plan, nbytes) == 1
    assert b"overlap" in lg.lib.logra_last_error()
    over = _sketch_group_targets(lg, shapes, r)
    over[1].S = over[0].S + 4 * (255 * 4 + 3)                    # the last element of target 0's S
    assert f(2, over, r, ws, wsb, plan, nbytes) == 1
    apart = _sketch_group_targets(lg, shapes, r)
    apart[1].S = apart[0].S + 4 * 256 * 4                        # just past it: no overlap
    assert f(2, apart, r, ws, wsb, plan, nbytes) in (0, 6)       # accepted (maps need the driver here)
    u = lg.lib.logra_sketch_accumulate_group
    empty = _sketch_group_targets(lg, [(0, 64, 64), (128, 0, 64)], r)
    assert f(2, empty, r, None, 0, plan, nbytes) == 0            # a plan (no maps needed)
    assert u(None, plan, None) == 1                              # no host plan
    assert u(plan, plan + 64, None) == 3                         # device copy misaligned
    zeros, zp = _aligned_buffer(nbytes)
    assert u(zp, zp, None) == 1                                  # not a plan


def test_row_stride_of_degenerate_tensors(lg):
    import torch

    rm = lg._binding._row_major
    assert rm(torch.empty((5, 12))[:, :8], "t") == 12
    assert rm(torch.empty((0, 1)).as_strided((0, 1), (1, 0)), "S") == 1      # torch's strides of an empty d×1
    assert rm(torch.empty((1, 16)).as_strided((1, 16), (3, 1)), "X") == 16   # one row: its stride is free
    assert rm(torch.empty((4, 8)).as_strided((4, 1), (8, 0)), "S") == 8      # one column: no inner stride
    with pytest.raises(ValueError):
        rm(torch.empty((4, 8)).t(), "X")
    with pytest.raises(ValueError):
        rm(torch.empty(8), "X")
