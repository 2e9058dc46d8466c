"""Vocabulary-parallel path on one GPU: the shards run one after another through
flce_shard_stats -> flce_combine_shards -> flce_backward (per shard) and must match the
whole-vocabulary fp64 oracle (tolerances as in the other parity tests); the shards'
dhidden terms come back in fp32 (dhidden_fp32) and are summed before one rounding, as
the all-reduce of the multi-GPU path sums them; the single-rank autograd wrapper must
match the unsharded entry points."""
import dataclasses

import numpy as np
import pytest
import torch

from linear_cross_entropy_forward_gb300 import (flce_backward, flce_combine_shards,
                                                flce_forward, flce_shard_stats,
                                                vocab_parallel_linear_cross_entropy)
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
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


CASES = [
    ("none_3shards", dataclasses.replace(wl.TINY, name="vp1", N=300, H=200, V=1000,
                                         reduction="none", grad_mode="normal"),
     [0, 256, 648, 1000], "hv"),
    ("mean_zloss_cap", dataclasses.replace(wl.TINY, name="vp2", N=384, H=256, V=2048, w_std=0.2,
                                           zloss_coef=1e-3, softcap=4.0),
     [0, 1024, 2048], "hv"),
    ("sum_vh_4shards", dataclasses.replace(wl.TINY, name="vp3", N=260, H=128, V=776,
                                           reduction="sum"),
     [0, 200, 392, 584, 776], "vh"),
    # eight uneven shards, ragged in every dimension
    ("mean_8shards", dataclasses.replace(wl.TINY, name="vp5", N=520, H=192, V=4104,
                                         zloss_coef=1e-3),
     [0, 8, 520, 1032, 1800, 2056, 3080, 3600, 4104], "hv"),
    ("none_vh_8shards_cap", dataclasses.replace(wl.TINY, name="vp6", N=300, H=128, V=2048,
                                                reduction="none", grad_mode="normal",
                                                w_std=0.2, softcap=5.0),
     [0, 256, 512, 768, 1024, 1280, 1536, 1792, 2048], "vh"),
]


@pytest.mark.parametrize("name,w,cuts,layout", CASES, ids=[c[0] for c in CASES])
def test_sequential_shards_match_oracle(name, w, cuts, layout):
    _cuda_or_skip()
    check_shards(w, cuts, layout)


def random_shard_case(i):
    """Random shapes (ragged in every dimension), 2-8 shards cut at random columns (on
    the 8-column grid a [H,V] shard's row stride needs; anywhere for [V,H]), and random
    reduction, z-loss, soft-cap and backward chunk."""
    import random
    r = random.Random(7000 + i)
    layout = r.choice(["hv", "vh"])
    reduction = r.choice(["none", "mean", "sum"])
    step = 8 if layout == "hv" else 1
    P = r.randint(2, 8)
    V = step * r.randint(P, 3000 // step)
    cuts = sorted(r.sample(range(1, V // step), P - 1))
    cuts = [0] + [c * step for c in cuts] + [V]
    w = dataclasses.replace(
        wl.TINY, name=f"vprand{i}", seed=300 + i,
        N=r.choice([1, 37, 255, 300, 513]), H=8 * r.randint(1, 48), V=V,
        reduction=reduction, ignore_frac=r.choice([0.0, 0.1, 0.5]),
        zloss_coef=r.choice([0.0, 1e-3]), softcap=r.choice([0.0, 0.0, 5.0]),
        w_std=r.choice([0.02, 0.2]), grad_mode="normal" if reduction == "none" else "ones")
    return w, cuts, layout, r.choice([0, 0, 256])


RANDOM_CASES = [random_shard_case(i) for i in range(12)]


@pytest.mark.parametrize("i", range(len(RANDOM_CASES)))
def test_random_shards_match_oracle(i):
    _cuda_or_skip()
    check_shards(*RANDOM_CASES[i])


def check_shards(w, cuts, layout, chunk_v=0):
    dev = torch.device("cuda")
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    hd, yd = hidden.to(dev), labels.to(dev)
    shards = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        ws = weight[:, a:b]
        shards.append((a, (ws if layout == "hv" else ws.t()).contiguous().to(dev)))
    stats = torch.stack([flce_shard_stats(hd, ws, yd, a, w.V, softcap=w.softcap,
                                          weight_layout=layout, validate=True)
                         for a, ws in shards])
    loss, ent, lse, ez = flce_combine_shards(stats, yd, w.V, w.reduction,
                                             zloss_coef=w.zloss_coef, H=w.H, validate=True)
    dh = torch.zeros(w.N, w.H, device=dev)
    dws = []
    for a, ws in shards:
        dhp, dwp = flce_backward(hd, ws, yd, lse, ez, g_loss.to(dev), g_ent.to(dev), w.reduction,
                                 zloss_coef=w.zloss_coef, softcap=w.softcap, validate=True,
                                 weight_layout=layout, v_offset=a, v_total=w.V,
                                 dhidden_fp32=True, chunk_v=chunk_v)
        assert dhp.dtype == torch.float32
        dh += dhp
        dws.append(dwp if layout == "hv" else dwp.t())
    dh = dh.to(torch.bfloat16)  # one rounding of the sum, as after the all-reduce
    dw = torch.cat(dws, dim=1)
    torch.cuda.synchronize()

    h64 = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W64 = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    y = labels.numpy()
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)
    o = orc.forward(h64, W64, y, w.reduction, **kw)
    dh_o, dw_o = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                              w.reduction, **kw)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    assert np.abs(f(lse) - o["lse"]).max() <= TOK_ABS
    assert np.abs(f(ez) - o["ez"]).max() <= TOK_ABS
    desc = f"{w} cuts={cuts} {layout} chunk_v={chunk_v}"
    if w.reduction == "none":
        assert np.abs(f(loss) - o["loss"]).max() <= TOK_ABS, desc
        assert np.abs(f(ent) - o["entropy"]).max() <= TOK_ABS, desc
    else:
        for got, want in ((loss.item(), o["loss"]), (ent.item(), o["entropy"])):
            assert (abs(got - want) <= RED_REL * abs(want)) if want != 0 else got == 0, desc
    for got, want in ((f(dh), dh_o), (f(dw), dw_o)):
        if np.linalg.norm(want) > 0:
            assert rel_l2(got, want) <= GRAD_REL_L2, desc
        else:  # every row ignored: exactly zero
            assert np.all(got == 0), desc


@pytest.mark.parametrize("V,layout", [(1024, "hv"), (1001, "vh")])
def test_single_rank_wrapper_matches_unsharded_path(V, layout):
    """Without a process group the wrapper is one shard holding the whole vocabulary:
    the same numbers as flce_forward / flce_backward (also for a [V,H] weight whose
    vocabulary is not a multiple of 8)."""
    _cuda_or_skip()
    dev = torch.device("cuda")
    w = dataclasses.replace(wl.TINY, name="vp4", N=256, H=128, V=V, zloss_coef=1e-3)
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    h = hidden.to(dev).requires_grad_(True)
    W = (weight if layout == "hv" else weight.t().contiguous()).to(dev).requires_grad_(True)
    y = labels.to(dev)
    loss, ent = vocab_parallel_linear_cross_entropy(h, W, y, 0, w.V, "mean", zloss_coef=1e-3,
                                                    weight_layout=layout)
    (loss + 0.25 * ent).backward()
    ref = flce_forward(h.detach(), W.detach(), y, "mean", zloss_coef=1e-3,
                       weight_layout=layout)
    assert abs(loss.item() - ref[0].item()) <= 1e-5 * abs(ref[0].item())
    assert abs(ent.item() - ref[1].item()) <= 1e-5 * abs(ref[1].item())
    dh, dw = flce_backward(h.detach(), W.detach(), y, ref[2], ref[3],
                           torch.ones(1, device=dev), torch.full((1,), 0.25, device=dev),
                           "mean", zloss_coef=1e-3, weight_layout=layout)
    assert rel_l2(h.grad.float().cpu().numpy(), dh.float().cpu().numpy()) <= 1e-3
    assert rel_l2(W.grad.float().cpu().numpy(), dw.float().cpu().numpy()) <= 1e-3


@pytest.mark.parametrize("V,chunk_v", [(1000, 0), (1000, 256), (70000, 0)])
def test_fp32_dhidden_rounds_to_the_bf16_dhidden(V, chunk_v):
    """dhidden_fp32 returns the fp32 accumulation the bf16 output is rounded from: one
    vocabulary chunk (the tile's accumulator, also over a 70000-column k-loop) or several
    (the fp32 sum over chunks), the same sums in the same order, so rounding it gives the
    bf16 output's bits."""
    _cuda_or_skip()
    dev = torch.device("cuda")
    w = dataclasses.replace(wl.TINY, name="vp7", N=300, H=136, V=V, zloss_coef=1e-3,
                            softcap=8.0)
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    _, _, lse, ez = flce_forward(hd, Wd, yd, w.reduction, zloss_coef=1e-3, softcap=8.0)
    kw = dict(zloss_coef=1e-3, softcap=8.0, chunk_v=chunk_v, validate=True)
    dh16, dw16 = flce_backward(hd, Wd, yd, lse, ez, g_loss.to(dev), g_ent.to(dev), w.reduction,
                               **kw)
    dh32, dw32 = flce_backward(hd, Wd, yd, lse, ez, g_loss.to(dev), g_ent.to(dev), w.reduction,
                               dhidden_fp32=True, **kw)
    torch.cuda.synchronize()
    assert dh32.dtype == torch.float32
    assert torch.equal(dh32.to(torch.bfloat16).view(torch.int16), dh16.view(torch.int16))
    assert torch.equal(dw32.view(torch.int16), dw16.view(torch.int16))
