"""flce_forward_noalloc: the forward pass for callers that cannot allocate device memory.

Some callers can't call cudaMalloc: their device memory is handed out up front by a
framework or serving runtime that keeps all of it, or they run under an allocator
they do not own, so they have no way to give flce_forward a workspace.
flce_forward_noalloc runs the same launch sequence on a static 64 MiB device array
instead.  These tests call it through the C ABI and check, on two calls in a row
(the second reuses what the first left in the array):
  - its outputs are bit for bit those of flce_forward, which runs the same kernels on
    a caller-provided workspace;
  - its outputs match the fp64 oracle within the tolerances of the other parity tests;
  - a problem larger than the array is refused with FLCE_ERR_SCRATCH_LIMIT before
    anything runs.
Each test builds its own inputs and outputs and depends on no other test, so the file
passes alone in a fresh process and after the rest of the suite.  It is named to be
collected last only so that, if it fails, a run that stops at the first failure
(pytest -x) has already run every other test.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOK_ABS = 2e-3
RED_REL = 1e-4
SCRATCH_LIMIT = 9  # FLCE_ERR_SCRATCH_LIMIT


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


CASES = [("none", 0.0, 0.0), ("mean", 1e-4, 30.0)]


@pytest.mark.parametrize("reduction,zc,cap", CASES)
def test_noalloc_forward_is_bitwise_the_regular_forward_and_matches_the_oracle(reduction, zc,
                                                                               cap):
    lib = _lib()
    from linear_cross_entropy_forward_gb300 import flce_forward, make_params
    from linear_cross_entropy_forward_gb300 import workloads as wl
    from oracle import flce_oracle as orc
    # several row and vocabulary tiles, ragged in both (1000 = 3 x 256 + 232 rows,
    # 8000 = 31 x 256 + 64 columns)
    w = dataclasses.replace(wl.TINY, name="noalloc", N=1000, H=512, V=8000,
                            reduction=reduction, zloss_coef=zc, softcap=cap)
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    dev = torch.device("cuda")
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    ref = flce_forward(hd, Wd, yd, reduction, zloss_coef=zc, softcap=cap, validate=True)
    torch.cuda.synchronize()
    o = orc.forward(orc.bf16_bits_to_f64(wl.bf16_bits(hidden)),
                    orc.bf16_bits_to_f64(wl.bf16_bits(weight)), labels.numpy(), reduction,
                    zloss_coef=zc, softcap=cap)
    p = make_params(w.N, w.H, w.V, reduction, zloss_coef=zc, softcap=cap, validate=True)
    n_out = w.N if reduction == "none" else 1
    for _ in range(2):  # the second call reuses the array the first one left behind
        rc, loss, ent, lse, ez = _noalloc(lib, p, hd, Wd, yd, n_out)
        assert rc == 0, lib.flce_strerror(rc)
        # the same kernels in the same order: the same bits
        for got, want in zip((loss, ent, lse, ez), ref):
            assert torch.equal(got, want)
        # and the oracle's values within the parity tolerances
        f64 = lambda t: t.cpu().numpy().astype(np.float64)  # noqa: E731
        assert np.abs(f64(lse) - o["lse"]).max() <= TOK_ABS
        assert np.abs(f64(ez) - o["ez"]).max() <= TOK_ABS
        if reduction == "none":
            assert np.abs(f64(loss) - o["loss"]).max() <= TOK_ABS
            assert np.abs(f64(ent) - o["entropy"]).max() <= TOK_ABS
        else:
            assert abs(loss.item() - o["loss"]) <= RED_REL * abs(o["loss"])
            assert abs(ent.item() - o["entropy"]) <= RED_REL * abs(o["entropy"])


def test_noalloc_refuses_problems_beyond_the_array():
    lib = _lib()
    from linear_cross_entropy_forward_gb300 import make_params, workspace_size
    p = make_params(16384, 3584, 152064, "none")  # the Qwen2.5 batch shape
    assert workspace_size(p, 0) > (64 << 20)
    dev = torch.device("cuda")
    sentinel = torch.full((16,), 7.0, device=dev)
    ptr = ctypes.c_void_p(sentinel.data_ptr())
    rc = lib.flce_forward_noalloc(ctypes.byref(p), ptr, ptr, ptr, ptr, ptr, ptr, ptr,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == SCRATCH_LIMIT
    assert b"64 MiB" in lib.flce_strerror(SCRATCH_LIMIT)
    # refused before anything was enqueued: the buffers passed in are untouched
    assert torch.all(sentinel == 7.0)
