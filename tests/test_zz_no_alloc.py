"""The allocation-free predicted-KL entry point, called through the C ABI.

logra_predicted_kl_noalloc exists for callers that cannot give the library
device memory where they need q(D): an engine whose device memory all belongs
to its own pool, or a C controller holding nothing but the logits pointers.
Its scratch is a fixed array inside the library, shared by every call, so the
checks here are that it agrees with logra_predicted_kl (which takes a
workspace) on two calls in a row with different inputs, and that it refuses
more rows than the array holds.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu

Q_TOL = 1e-4  # the relative tolerance the KL parity tests use
DEV = "cuda"


@pytest.fixture(scope="module")
def lg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_gradient_sketching_gb300 as mod

    torch.cuda.set_device(0)
    return mod


def _call_noalloc(lg, cur, prop, tau, mask, q, row_kl):
    dtype = 0 if cur.dtype == torch.bfloat16 else 1
    stream = torch.cuda.current_stream().cuda_stream
    return lg.lib.logra_predicted_kl_noalloc(
        ctypes.c_void_p(cur.data_ptr()), ctypes.c_void_p(prop.data_ptr()), dtype, cur.shape[0], cur.shape[1],
        cur.stride(0), ctypes.c_float(tau), None if mask is None else ctypes.c_void_p(mask.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(row_kl.data_ptr()), ctypes.c_void_p(stream))


def _compare(lg, cur, prop, tau=1.0, mask=None):
    rows = cur.shape[0]
    q_na = torch.full((), -1.0, dtype=torch.float64, device=DEV)
    rk_na = torch.full((rows,), -1.0, dtype=torch.float32, device=DEV)
    assert _call_noalloc(lg, cur, prop, tau, mask, q_na, rk_na) == 0, lg.logra_last_error()
    rk_ws = torch.empty(rows, dtype=torch.float32, device=DEV)
    q_ws = lg.logra_predicted_kl(cur, prop, tau, row_mask=mask, row_kl_out=rk_ws)
    torch.cuda.synchronize()
    assert lg.logra_device_error() == 0
    q_a, q_b = float(q_na.item()), float(q_ws.item())
    assert q_b > 0 and abs(q_a - q_b) <= Q_TOL * q_b, (q_a, q_b)
    a, b = rk_na.double().cpu().numpy(), rk_ws.double().cpu().numpy()
    assert np.allclose(a, b, rtol=Q_TOL, atol=0)
    return q_a


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(lg):
    # First call: 300 full-vocabulary bf16 rows.  Second call: fewer fp32 rows
    # with a mask, so stale per-row values from the first call would show.
    cur, prop = synthetic.kl_logits("qwen", 0.1, rows=300, device=DEV)
    q1 = _compare(lg, cur, prop)
    cur2, prop2 = synthetic.kl_logits("tiny", 0.05, device=DEV)
    mask = torch.tensor([1, 0] * 8, dtype=torch.uint8, device=DEV)
    q2 = _compare(lg, cur2, prop2, tau=0.8, mask=mask)
    assert q1 != q2


def test_noalloc_refuses_more_rows_than_it_holds(lg):
    rows = lg.LOGRA_KL_NOALLOC_MAX_ROWS + 1 if hasattr(lg, "LOGRA_KL_NOALLOC_MAX_ROWS") else 65537
    small = torch.zeros((1, 8), dtype=torch.float32, device=DEV)
    q = torch.zeros((), dtype=torch.float64, device=DEV)
    rk = torch.zeros(1, dtype=torch.float32, device=DEV)
    dtype = 1
    st = lg.lib.logra_predicted_kl_noalloc(ctypes.c_void_p(small.data_ptr()), ctypes.c_void_p(small.data_ptr()),
                                           dtype, rows, 8, 8, ctypes.c_float(1.0), None,
                                           ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(rk.data_ptr()), None)
    assert st == 5  # LOGRA_ERR_UNSUPPORTED, nothing launched
    assert "65536" in lg.logra_last_error()
