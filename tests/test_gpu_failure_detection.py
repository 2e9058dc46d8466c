"""Device-side failure detection without faulting the GPU: a bounded mbarrier wait that
nothing satisfies gives up after its limit, the error word in the workspace reports
FLCE_ERR_TIMEOUT through flce_status, and the CUDA context stays usable for the next
call (the same wait guards every stage, accumulator and drain barrier of the GEMMs)."""
import time

import numpy as np
import pytest
import torch

from linear_cross_entropy_forward_gb300 import _binding as B
from linear_cross_entropy_forward_gb300 import flce_forward, flce_status
from linear_cross_entropy_forward_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FLCE_ERR_TIMEOUT = 6


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


def test_bounded_wait_times_out_and_context_survives():
    _cuda_or_skip()
    t0 = time.time()
    assert B.selftest_wait_timeout(limit_ns=20_000_000) == FLCE_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    # the context is still usable: a forward right after runs and reports no error
    w = wl.TINY
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    dev = torch.device("cuda")
    ws = torch.empty(B.workspace_size(B.make_params(w.N, w.H, w.V, w.reduction), 0),
                     dtype=torch.uint8, device=dev)
    loss, ent, lse, ez = flce_forward(hidden.to(dev), weight.to(dev), labels.to(dev),
                                      w.reduction, workspace=ws)
    assert flce_status(ws) == 0
    assert np.isfinite(float(loss[0])) and np.isfinite(float(ent[0]))
    assert torch.isfinite(lse).all()


def test_timeout_status_is_per_workspace():
    """A timeout recorded in one workspace does not leak into another call's status."""
    _cuda_or_skip()
    assert B.selftest_wait_timeout(limit_ns=5_000_000) == FLCE_ERR_TIMEOUT
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert flce_status(ws) == 0
