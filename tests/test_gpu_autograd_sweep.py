"""Seeded random sweep of the autograd entry point linear_cross_entropy: random shapes
(ragged in every dimension) and options (reduction, z-loss, soft-cap, label smoothing,
class weights, weight layout, gradient in forward), random objectives built from its
two outputs, and the gradients autograd delivers to hidden and weight against the fp64
oracle's backward at the same upstream gradients (rel-L2 <= 1e-2; forward outputs
within the parity tolerances; ignored rows' dhidden exactly zero)."""
import dataclasses
import random

import numpy as np
import pytest
import torch

from linear_cross_entropy_forward_gb300 import linear_cross_entropy
from linear_cross_entropy_forward_gb300 import workloads as wl
from oracle import flce_oracle as orc

pytestmark = pytest.mark.gpu

TOK_ABS = 2e-3
RED_REL = 1e-4
GRAD_REL_L2 = 1e-2


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


def rel_l2(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def random_case(i):
    r = random.Random(9000 + i)
    layout = r.choice(["hv", "vh"])
    reduction = r.choice(["none", "mean", "sum"])
    V = r.randint(2, 3000) if layout == "vh" else 8 * r.randint(1, 375)
    w = dataclasses.replace(
        wl.TINY, name=f"ag{i}", seed=700 + i, N=r.choice([1, 37, 300, 513]),
        H=8 * r.randint(1, 48), V=V, reduction=reduction,
        ignore_frac=r.choice([0.0, 0.1, 0.5]), zloss_coef=r.choice([0.0, 1e-3]),
        softcap=r.choice([0.0, 0.0, 5.0]), w_std=r.choice([0.02, 0.2]))
    opts = dict(layout=layout, eps=r.choice([0.0, 0.0, 0.1]),
                class_weight=r.random() < 0.3,
                gif=reduction != "none" and r.random() < 0.4,
                loss_only=r.random() < 0.25,
                a=r.uniform(-2.0, 2.0), b=r.uniform(-1.0, 1.0))
    return w, opts


CASES = [random_case(i) for i in range(12)]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_autograd_gradients_match_oracle(i):
    _cuda_or_skip()
    w, o = CASES[i]
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    cw = None
    if o["class_weight"]:
        cw = (torch.rand(w.V, generator=torch.Generator().manual_seed(i)) + 0.5).float()
    dev = torch.device("cuda")
    h = hidden.to(dev).requires_grad_(True)
    Wsrc = weight if o["layout"] == "hv" else weight.t().contiguous()
    W = Wsrc.to(dev).requires_grad_(True)
    y = labels.to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, weight_layout=o["layout"],
              label_smoothing=o["eps"], class_weight=None if cw is None else cw.to(dev))
    gen = torch.Generator().manual_seed(100 + i)
    if o["gif"]:
        # objective a * (loss + c * entropy), c fixed at forward time
        loss, ent = linear_cross_entropy(h, W, y, w.reduction, grad_in_forward=True,
                                         entropy_coef=o["b"], **kw)
        (o["a"] * loss).backward()
        gl = np.array([o["a"]])
        ge = np.array([o["a"] * o["b"]])
    else:
        loss, ent = linear_cross_entropy(h, W, y, w.reduction, **kw)
        if w.reduction == "none":
            a = torch.randn(w.N, generator=gen)
            b = torch.randn(w.N, generator=gen)
            obj = (a.to(dev) * loss).sum()
            if not o["loss_only"]:
                obj = obj + (b.to(dev) * ent).sum()
            gl = a.numpy().astype(np.float64)
            ge = np.zeros(w.N) if o["loss_only"] else b.numpy().astype(np.float64)
        else:
            obj = o["a"] * loss if o["loss_only"] else o["a"] * loss + o["b"] * ent
            gl = np.array([o["a"]])
            ge = np.array([0.0 if o["loss_only"] else o["b"]])
        obj.backward()
    torch.cuda.synchronize()

    h64 = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W64 = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    yn = labels.numpy()
    okw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, label_smoothing=o["eps"],
               class_weight=None if cw is None else cw.numpy())
    ref = orc.forward(h64, W64, yn, w.reduction, **okw)
    dh_o, dw_o = orc.backward(h64, W64, yn, ref["lse"], ref["ez"], gl, ge, w.reduction, **okw)
    desc = f"case {i}: {w} {o}"
    if w.reduction == "none":
        assert np.abs(f64(loss) - ref["loss"]).max() <= TOK_ABS, desc
        assert np.abs(f64(ent) - ref["entropy"]).max() <= TOK_ABS, desc
    else:
        for got, want in ((float(loss.detach()), float(ref["loss"])),
                          (float(ent.detach()), float(ref["entropy"]))):
            assert (abs(got - want) <= RED_REL * abs(want)) if want != 0 else got == 0, desc
    dw_got = f64(W.grad) if o["layout"] == "hv" else f64(W.grad).T
    for got, want in ((f64(h.grad), dh_o), (dw_got, dw_o)):
        if np.linalg.norm(want) > 0:
            assert rel_l2(got, want) <= GRAD_REL_L2, desc
        else:
            assert np.all(got == 0), desc
    ign = np.nonzero(~ref["valid"])[0]
    if ign.size:
        assert torch.all(h.grad.detach().cpu()[torch.from_numpy(ign)].view(torch.int16) == 0), desc
