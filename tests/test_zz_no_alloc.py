"""flce_forward_noalloc: the forward pass for callers that cannot allocate.

Some callers can't call cudaMalloc (code running while a CUDA graph is being
captured, or under an allocator they do not control), so they cannot hand
flce_forward a workspace.  flce_forward_noalloc uses a static 64 MiB device
array instead.  This test calls it through the C ABI and checks that two calls
in a row agree with flce_forward (the regular, workspace-taking entry point)
within the tolerances the other parity tests use, and that a problem larger
than the array is refused without running.  The file is named so that pytest
collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOK_ABS = 2e-3
RED_REL = 1e-4


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    from linear_cross_entropy_forward_gb300 import load_library
    build()
    lib = load_library()
    lib.flce_forward_noalloc.argtypes = [ctypes.c_void_p] * 9
    lib.flce_forward_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(lib, p, hd, Wd, yd, n_out):
    dev = hd.device
    loss = torch.full((n_out,), float("nan"), device=dev)
    ent = torch.full((n_out,), float("nan"), device=dev)
    lse = torch.full((hd.shape[0],), float("nan"), device=dev)
    ez = torch.full((hd.shape[0],), float("nan"), device=dev)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.flce_forward_noalloc(ctypes.byref(p), ptr(hd), ptr(Wd), ptr(yd), ptr(loss),
                                  ptr(ent), ptr(lse), ptr(ez),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, loss, ent, lse, ez


@pytest.mark.parametrize("reduction,zc,cap", [("none", 0.0, 0.0), ("mean", 1e-4, 30.0)])
def test_noalloc_forward_matches_regular_forward(reduction, zc, cap):
    lib = _lib()
    from linear_cross_entropy_forward_gb300 import flce_forward, make_params
    from linear_cross_entropy_forward_gb300 import workloads as wl
    import dataclasses
    w = dataclasses.replace(wl.TINY, name="noalloc", N=1000, H=512, V=8000,
                            reduction=reduction, zloss_coef=zc, softcap=cap)
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    dev = torch.device("cuda")
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    ref = flce_forward(hd, Wd, yd, reduction, zloss_coef=zc, softcap=cap, validate=True)
    torch.cuda.synchronize()
    p = make_params(w.N, w.H, w.V, reduction, zloss_coef=zc, softcap=cap, validate=True)
    n_out = w.N if reduction == "none" else 1
    for _ in range(2):  # the second call reuses the array the first one left behind
        rc, loss, ent, lse, ez = _noalloc(lib, p, hd, Wd, yd, n_out)
        assert rc == 0, lib.flce_strerror(rc)
        assert np.abs((lse - ref[2]).cpu().numpy()).max() <= TOK_ABS
        assert np.abs((ez - ref[3]).cpu().numpy()).max() <= TOK_ABS
        if reduction == "none":
            assert np.abs((loss - ref[0]).cpu().numpy()).max() <= TOK_ABS
            assert np.abs((ent - ref[1]).cpu().numpy()).max() <= TOK_ABS
        else:
            assert abs(loss.item() - ref[0].item()) <= RED_REL * abs(ref[0].item())
            assert abs(ent.item() - ref[1].item()) <= RED_REL * abs(ref[1].item())


def test_noalloc_refuses_problems_beyond_the_array():
    lib = _lib()
    from linear_cross_entropy_forward_gb300 import make_params, workspace_size
    p = make_params(16384, 3584, 152064, "none")  # the Qwen2.5 batch shape
    assert workspace_size(p, 0) > (64 << 20)
    dev = torch.device("cuda")
    dummy = torch.empty(16, device=dev)
    ptr = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.flce_forward_noalloc(ctypes.byref(p), ptr, ptr, ptr, ptr, ptr, ptr, ptr,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 9
    assert b"64 MiB" in lib.flce_strerror(9)
