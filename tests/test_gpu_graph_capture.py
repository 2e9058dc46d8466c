"""The forward + backward step enqueues only kernels and memsets on the caller's stream
(workspaces are caller-owned), so it can be captured in a CUDA graph after one eager
call (which caches the device queries); replays give the eager results bit for bit."""
import dataclasses

import pytest
import torch

from linear_cross_entropy_forward_gb300 import flce_backward, flce_forward, flce_forward_backward
from linear_cross_entropy_forward_gb300 import make_params, workspace_size
from linear_cross_entropy_forward_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


@pytest.mark.parametrize("fused", [False, True], ids=["two_call", "grad_in_forward"])
def test_step_replays_from_a_cuda_graph(fused):
    _cuda_or_skip()
    w = dataclasses.replace(wl.TINY, name="g", N=700, H=256, V=1536, zloss_coef=1e-3)
    h, W, y, gl, ge = wl.make_inputs(w)
    dev = torch.device("cuda")
    hd, Wd, yd, gld, ged = h.to(dev), W.to(dev), y.to(dev), gl.to(dev), ge.to(dev)
    p = make_params(w.N, w.H, w.V, w.reduction, zloss_coef=w.zloss_coef)
    outs = dict(loss=torch.empty(1, device=dev), ent=torch.empty(1, device=dev),
                lse=torch.empty(w.N, device=dev), ez=torch.empty(w.N, device=dev),
                dh=torch.empty(w.N, w.H, dtype=torch.bfloat16, device=dev),
                dw=torch.empty(w.H, w.V, dtype=torch.bfloat16, device=dev))
    if fused:
        ws = [torch.empty(workspace_size(p, 3), dtype=torch.uint8, device=dev)]
    else:
        ws = [torch.empty(workspace_size(p, 0), dtype=torch.uint8, device=dev),
              torch.empty(workspace_size(p, 1), dtype=torch.uint8, device=dev)]
    kw = dict(zloss_coef=w.zloss_coef)

    def step(stream):
        o = outs
        if fused:
            flce_forward_backward(hd, Wd, yd, gld, ged, w.reduction, workspace=ws[0], stream=stream,
                                  out=(o["loss"], o["ent"], o["lse"], o["ez"], o["dh"], o["dw"]),
                                  **kw)
        else:
            flce_forward(hd, Wd, yd, w.reduction, workspace=ws[0], stream=stream,
                         out=(o["loss"], o["ent"], o["lse"], o["ez"]), **kw)
            flce_backward(hd, Wd, yd, o["lse"], o["ez"], gld, ged, w.reduction, workspace=ws[1],
                          stream=stream, out=(o["dh"], o["dw"]), **kw)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in outs.items()}
    for v in outs.values():
        v.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for k, v in outs.items():
        assert torch.equal(v.view(torch.int16) if v.dtype == torch.bfloat16 else v,
                           eager[k].view(torch.int16) if v.dtype == torch.bfloat16 else eager[k]), k
