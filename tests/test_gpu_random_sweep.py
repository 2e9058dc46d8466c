"""Seeded random sweep: small problems with random shapes (ragged in every dimension)
and random combinations of every option -- reduction, z-loss, soft-cap, label
smoothing, class weights, weight layout, backward vocabulary chunk, token chunk, and
the two-call vs gradient-in-forward path -- against the fp64 oracle, with the stated
tolerances (per-token abs <= 2e-3, reduced rel <= 1e-4, gradients rel-L2 <= 1e-2,
ignored rows exactly zero).  A second set adds the options of the C ABI's later
version: a [V,H] weight with any vocabulary size, and an fp32 dhidden.  A third set
takes medium shapes (thousands of tiles per GEMM, several chunks)."""
import dataclasses
import random

import numpy as np
import pytest
import torch

from linear_cross_entropy_forward_gb300 import (flce_backward, flce_forward,
                                                flce_forward_backward)
from linear_cross_entropy_forward_gb300 import workloads as wl
from oracle import flce_oracle as orc

pytestmark = pytest.mark.gpu

TOK_ABS = 2e-3
RED_REL = 1e-4
GRAD_REL_L2 = 1e-2
N_CASES = 32


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


def rel_l2(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def random_case(i):
    r = random.Random(1000 + i)
    reduction = r.choice(["none", "mean", "sum"])
    w = dataclasses.replace(
        wl.TINY, name=f"rand{i}", seed=50 + i,
        N=r.choice([1, 37, 128, 255, 300, 513, 777, 1100]),
        H=8 * r.randint(1, 80),
        V=8 * r.randint(1, 500),
        reduction=reduction,
        ignore_frac=r.choice([0.0, 0.1, 0.5]),
        zloss_coef=r.choice([0.0, 0.0, 1e-3, 1e-2]),
        softcap=r.choice([0.0, 0.0, 5.0, 30.0]),
        w_std=r.choice([0.02, 0.1, 0.3]),
        grad_mode="normal" if reduction == "none" else "ones")
    opts = dict(
        eps=r.choice([0.0, 0.0, 0.1]),
        class_weight=r.random() < 0.3,
        layout=r.choice(["hv", "vh"]),
        chunk_v=r.choice([0, 0, 256, 512]),
        fused=r.random() < 0.5,
        chunk_n=r.choice([0, 512]))
    return w, opts


CASES = [random_case(i) for i in range(N_CASES)]
N_CASES2 = 16


def random_case_v2(i):
    """[V,H] weights with any vocabulary size (not a multiple of 8) and fp32 dhidden,
    with the other options drawn as above."""
    w, o = random_case(100 + i)
    r = random.Random(5000 + i)
    o = dict(o, layout="vh", dh32=r.random() < 0.6)
    w = dataclasses.replace(w, name=f"rand2_{i}", V=r.randint(1, 4000))
    return w, o


CASES2 = [random_case_v2(i) for i in range(N_CASES2)]
N_CASES3 = 8


def random_case_medium(i):
    """Medium shapes: thousands of output tiles, so every pair of the persistent GEMMs
    takes many tiles from the dynamic schedule, with several backward vocabulary chunks
    or token chunks; the other options drawn as above."""
    w, o = random_case(200 + i)
    r = random.Random(8000 + i)
    V = 8 * r.randint(500, 5000) if o["layout"] == "hv" else r.randint(4000, 40000)
    w = dataclasses.replace(w, name=f"rand3_{i}", N=r.randint(1000, 5000),
                            H=8 * r.randint(16, 256), V=V)
    o = dict(o, chunk_v=r.choice([0, 2048, 8192]), chunk_n=r.choice([0, 1024]))
    return w, o


CASES3 = [random_case_medium(i) for i in range(N_CASES3)]


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(i):
    _cuda_or_skip()
    check_case(i, *CASES[i])


@pytest.mark.parametrize("i", range(N_CASES2))
def test_random_case_any_vocabulary_and_fp32_dhidden(i):
    _cuda_or_skip()
    check_case(1000 + i, *CASES2[i])


@pytest.mark.parametrize("i", range(N_CASES3))
def test_random_medium_case_matches_oracle(i):
    _cuda_or_skip()
    check_case(2000 + i, *CASES3[i])


def check_case(i, w, o):
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    cw = None
    if o["class_weight"]:
        cw = (torch.rand(w.V, generator=torch.Generator().manual_seed(i)) + 0.5).float()
    h = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    y = labels.numpy()
    okw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, label_smoothing=o["eps"],
               class_weight=None if cw is None else cw.numpy())
    ref = orc.forward(h, W, y, w.reduction, **okw)
    dh_o, dw_o = orc.backward(h, W, y, ref["lse"], ref["ez"], g_loss.numpy(), g_ent.numpy(),
                              w.reduction, **okw)

    dev = torch.device("cuda")
    hd, yd, gl, ge = hidden.to(dev), labels.to(dev), g_loss.to(dev), g_ent.to(dev)
    Wd = weight.to(dev) if o["layout"] == "hv" else weight.t().contiguous().to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, weight_layout=o["layout"],
              label_smoothing=o["eps"], class_weight=None if cw is None else cw.to(dev))
    dh32 = o.get("dh32", False)
    if o["fused"]:
        loss, ent, lse, ez, dh, dw = flce_forward_backward(
            hd, Wd, yd, gl, ge, w.reduction, validate=True, chunk_n=o["chunk_n"],
            dhidden_fp32=dh32, **kw)
    else:
        loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, validate=True, **kw)
        dh, dw = flce_backward(hd, Wd, yd, lse, ez, gl, ge, w.reduction, validate=True,
                               chunk_v=o["chunk_v"], dhidden_fp32=dh32, **kw)
    assert dh.dtype == (torch.float32 if dh32 else torch.bfloat16)
    torch.cuda.synchronize()
    if o["layout"] == "vh":
        dw = dw.t()
    valid = ref["valid"]
    desc = f"case {i}: {w} {o}"
    assert np.abs(f64(lse) - ref["lse"]).max() <= TOK_ABS, desc
    assert np.abs(f64(ez) - ref["ez"]).max() <= TOK_ABS, desc
    if w.reduction == "none":
        assert np.abs(f64(loss) - ref["loss"]).max() <= TOK_ABS, desc
        assert np.abs(f64(ent) - ref["entropy"]).max() <= TOK_ABS, desc
        assert np.all(f64(loss)[~valid] == 0) and np.all(f64(ent)[~valid] == 0), desc
    else:
        for got, want in ((float(loss[0]), float(ref["loss"])),
                          (float(ent[0]), float(ref["entropy"]))):
            assert (abs(got - want) <= RED_REL * abs(want)) if want != 0 else got == 0, desc
    for got, want in ((f64(dh), dh_o), (f64(dw), dw_o)):
        if np.linalg.norm(want) > 0:
            assert rel_l2(got, want) <= GRAD_REL_L2, desc
        else:  # every row ignored (or zero upstream gradients): exactly zero
            assert np.all(got == 0), desc
    ign = np.nonzero(~valid)[0]
    if ign.size:  # bitwise zero (no -0.0 either)
        bits = dh.cpu()[torch.from_numpy(ign)].view(torch.int32 if dh32 else torch.int16)
        assert torch.all(bits == 0), desc
