"""Steps whose inputs come from pinned host memory, with the copies overlapped.

A training or evaluation loop that keeps its batches on the host pays a host-to-device
copy per step (for an LM head, mostly the weight).  HostPipeline double-buffers the
device inputs: the copies of step i+1 run on a side stream while step i computes on
the current stream, and each step's loss and entropy are copied back into pinned host
memory.  Plumbing only (buffers, streams, events); the computation is the library's
flce_forward + flce_backward, or flce_forward_backward with grad_in_forward=True.
"""
from __future__ import annotations

import torch

from ._binding import (flce_backward, flce_forward, flce_forward_backward, make_params,
                       workspace_size)
from .workloads import IGNORE_INDEX, RED_NONE, reduction_code


class HostPipeline:
    """fwd + bwd steps on inputs in pinned host memory.

    submit(hidden, weight, labels, g_loss, g_entropy) enqueues the host-to-device copy
    of one step's inputs (all pinned CPU tensors of the step's shapes) on the copy
    stream; step() runs the oldest submitted step on the current stream and enqueues
    the device-to-host copy of its loss and entropy, returning the pinned host tensors
    that receive them (valid once the stream has reached them).  Submitting step i+1
    before calling step() for step i overlaps the copy with the computation; at most
    two steps can be submitted and not yet run.
    """

    def __init__(self, N, H, V, reduction="mean", ignore_index=IGNORE_INDEX, zloss_coef=0.0,
                 softcap=0.0, weight_layout="hv", grad_in_forward=False, device=None):
        self.dev = torch.device("cuda") if device is None else torch.device(device)
        self.N, self.H, self.V = N, H, V
        self.reduction = reduction
        self.kw = dict(ignore_index=ignore_index, zloss_coef=zloss_coef, softcap=softcap,
                       weight_layout=weight_layout)
        self.grad_in_forward = grad_in_forward
        wshape = (H, V) if weight_layout == "hv" else (V, H)
        n_out = N if reduction_code(reduction) == RED_NONE else 1
        dev = self.dev

        def inputs():
            return dict(hidden=torch.empty(N, H, dtype=torch.bfloat16, device=dev),
                        weight=torch.empty(wshape, dtype=torch.bfloat16, device=dev),
                        labels=torch.empty(N, dtype=torch.int64, device=dev),
                        g_loss=torch.empty(n_out, dtype=torch.float32, device=dev),
                        g_entropy=torch.empty(n_out, dtype=torch.float32, device=dev))

        self.bufs = [inputs(), inputs()]
        self.copied = [torch.cuda.Event(), torch.cuda.Event()]
        self.consumed = [torch.cuda.Event(), torch.cuda.Event()]
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.loss = torch.empty(n_out, dtype=torch.float32, device=dev)
        self.ent = torch.empty(n_out, dtype=torch.float32, device=dev)
        self.lse = torch.empty(N, dtype=torch.float32, device=dev)
        self.ez = torch.empty(N, dtype=torch.float32, device=dev)
        self.dh = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty(wshape, dtype=torch.bfloat16, device=dev)
        p = make_params(N, H, V, reduction, ignore_index, zloss_coef, softcap,
                        weight_layout=weight_layout)
        if grad_in_forward:
            self.ws = [torch.empty(workspace_size(p, 3), dtype=torch.uint8, device=dev)]
        else:
            self.ws = [torch.empty(workspace_size(p, 0), dtype=torch.uint8, device=dev),
                       torch.empty(workspace_size(p, 1), dtype=torch.uint8, device=dev)]
        self.loss_h = torch.empty(n_out, dtype=torch.float32).pin_memory()
        self.ent_h = torch.empty(n_out, dtype=torch.float32).pin_memory()
        self.n_submitted = 0
        self.n_run = 0

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.bufs[0].values())

    def d2h_bytes(self) -> int:
        return 2 * self.loss.numel() * 4

    def submit(self, hidden, weight, labels, g_loss, g_entropy):
        if self.n_submitted - self.n_run >= 2:
            raise RuntimeError("two steps are already waiting: call step() first")
        b = self.n_submitted % 2
        buf = self.bufs[b]
        with torch.cuda.stream(self.copy_stream):
            # the buffer's previous step must have finished reading it
            self.copy_stream.wait_event(self.consumed[b])
            for name, src in (("hidden", hidden), ("weight", weight), ("labels", labels),
                              ("g_loss", g_loss), ("g_entropy", g_entropy)):
                buf[name].copy_(src, non_blocking=True)
            self.copied[b].record(self.copy_stream)
        self.n_submitted += 1

    def step(self):
        if self.n_run >= self.n_submitted:
            raise RuntimeError("no submitted step to run")
        b = self.n_run % 2
        buf = self.bufs[b]
        stream = torch.cuda.current_stream(self.dev)
        stream.wait_event(self.copied[b])
        if self.grad_in_forward:
            flce_forward_backward(buf["hidden"], buf["weight"], buf["labels"], buf["g_loss"],
                                  buf["g_entropy"], self.reduction, workspace=self.ws[0],
                                  out=(self.loss, self.ent, self.lse, self.ez, self.dh,
                                       self.dw), **self.kw)
        else:
            flce_forward(buf["hidden"], buf["weight"], buf["labels"], self.reduction,
                         workspace=self.ws[0], out=(self.loss, self.ent, self.lse, self.ez),
                         **self.kw)
            flce_backward(buf["hidden"], buf["weight"], buf["labels"], self.lse, self.ez,
                          buf["g_loss"], buf["g_entropy"], self.reduction, workspace=self.ws[1],
                          out=(self.dh, self.dw), **self.kw)
        self.consumed[b].record(stream)
        self.loss_h.copy_(self.loss, non_blocking=True)
        self.ent_h.copy_(self.ent, non_blocking=True)
        self.n_run += 1
        return self.loss_h, self.ent_h
