"""HostPipeline: steps on pinned host inputs with double-buffered, overlapped copies
give exactly what the direct calls give on the same inputs (same kernels, same data)."""
import dataclasses

import pytest
import torch

from linear_cross_entropy_forward_gb300 import (HostPipeline, flce_backward, flce_forward,
                                                flce_forward_backward)
from linear_cross_entropy_forward_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


@pytest.mark.parametrize("gif", [False, True], ids=["two_call", "grad_in_forward"])
@pytest.mark.parametrize("layout", ["hv", "vh"])
def test_pipeline_steps_match_direct_calls(gif, layout):
    """[H,V] weights, and [V,H] ones with an odd vocabulary and a soft-cap."""
    _cuda_or_skip()
    base = dataclasses.replace(wl.TINY, name="p", N=700, H=256, V=1536, zloss_coef=1e-3)
    if layout == "vh":
        base = dataclasses.replace(base, V=1537, softcap=5.0, w_std=0.2)
    steps = [wl.make_inputs(dataclasses.replace(base, seed=s)) for s in (11, 12, 13, 14)]
    if layout == "vh":
        steps = [(h, W.t().contiguous(), y, gl, ge) for h, W, y, gl, ge in steps]
    kw = dict(zloss_coef=base.zloss_coef, softcap=base.softcap, weight_layout=layout)
    pipe = HostPipeline(base.N, base.H, base.V, base.reduction, grad_in_forward=gif, **kw)
    pinned = [tuple(t.pin_memory() for t in st) for st in steps]
    got = []
    pipe.submit(*pinned[0])
    for i in range(len(pinned)):
        if i + 1 < len(pinned):
            pipe.submit(*pinned[i + 1])
        loss_h, ent_h = pipe.step()
        torch.cuda.synchronize()
        got.append((loss_h.clone(), ent_h.clone()))
    dh_last, dw_last = pipe.dh.clone(), pipe.dw.clone()
    with pytest.raises(RuntimeError):
        pipe.step()
    dev = torch.device("cuda")
    for (h, W, y, gl, ge), (loss_h, ent_h) in zip(steps, got):
        hd, Wd, yd = h.to(dev), W.to(dev), y.to(dev)
        loss, ent, lse, ez = flce_forward(hd, Wd, yd, base.reduction, **kw)
        assert torch.equal(loss.cpu(), loss_h) and torch.equal(ent.cpu(), ent_h)
    if gif:
        *_, dh, dw = flce_forward_backward(hd, Wd, yd, gl.to(dev), ge.to(dev), base.reduction,
                                           **kw)
    else:
        dh, dw = flce_backward(hd, Wd, yd, lse, ez, gl.to(dev), ge.to(dev), base.reduction,
                               **kw)
    assert torch.equal(dh.view(torch.int16), dh_last.view(torch.int16))
    assert torch.equal(dw.view(torch.int16), dw_last.view(torch.int16))


def test_pipeline_refuses_a_third_pending_step():
    _cuda_or_skip()
    w = dataclasses.replace(wl.TINY, name="p2", N=64, H=64, V=256)
    pipe = HostPipeline(w.N, w.H, w.V, w.reduction)
    ins = tuple(t.pin_memory() for t in wl.make_inputs(w))
    pipe.submit(*ins)
    pipe.submit(*ins)
    with pytest.raises(RuntimeError):
        pipe.submit(*ins)
    pipe.step()
    pipe.submit(*ins)
    torch.cuda.synchronize()
