"""Failure reporting: a bounded wait that runs out is reported through the
device error word and leaves the context usable (no fault, no hang)."""

import numpy as np
import pytest
import torch

import synthetic
from oracle import philox as oph
from oracle import sketch as osk

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


def test_wait_limit_reports_and_context_survives(lg):
    assert lg.logra_device_error() == 0
    lg.logra_self_test_wait_timeout()
    assert lg.logra_device_error() == 7          # the code of the self-test wait
    assert lg.logra_device_error() == 0          # reading cleared it
    # the context still runs the real path correctly
    d, k, r, T = 256, 256, 16, 128
    X, dY = synthetic.microbatch("tiny", 0, "ft", 0, T, d, k, DEV)
    S = torch.zeros((d, r), device=DEV)
    lg.logra_sketch_accumulate(X, dY, S, 3, 1, r)
    torch.cuda.synchronize()
    assert lg.logra_device_error() == 0
    ref = osk.sketch_accumulate(np.zeros((d, r)), [(X.double().cpu().numpy(), dY.double().cpu().numpy())],
                                oph.projection(3, 1, r, k))
    assert np.linalg.norm(S.double().cpu().numpy() - ref) / np.linalg.norm(ref) <= 1e-3
