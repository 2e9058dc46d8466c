"""GPU parity of the gradient-in-forward path (flce_forward_backward, Liger-Kernel
PR #551's "gradient in forward"): one call computes loss, entropy, dhidden and dweight
from logits it keeps per token chunk, without the backward's recompute.

Checked against the fp64 oracle with the two-call path's tolerances (per-token abs
<= 2e-3, reduced rel <= 1e-4, gradients rel-L2 <= 1e-2, ignored rows exactly 0), and
against the two-call path itself: the forward statistics are the same kernels'
(bitwise equal), the dlogits are formed by the same per-element arithmetic from the
same fp32 accumulators, so with one token chunk dweight agrees bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

import _fullsize_oracle as fso
from linear_cross_entropy_forward_gb300 import (flce_backward, flce_forward,
                                                flce_forward_backward, flce_scale_bf16,
                                                linear_cross_entropy)
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
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _kw(w, layout, eps, cw):
    return dict(zloss_coef=w.zloss_coef, softcap=w.softcap, weight_layout=layout,
                label_smoothing=eps, class_weight=cw)


def run_fused(w, hidden, weight, labels, g_loss, g_ent, chunk_n=0, layout="hv", eps=0.0,
              cw=None):
    dev = torch.device("cuda")
    hd, yd = hidden.to(dev), labels.to(dev)
    Wd = weight.to(dev) if layout == "hv" else weight.t().contiguous().to(dev)
    cwd = None if cw is None else cw.to(dev)
    out = flce_forward_backward(hd, Wd, yd, g_loss.to(dev), g_ent.to(dev), w.reduction,
                                validate=True, chunk_n=chunk_n, **_kw(w, layout, eps, cwd))
    torch.cuda.synchronize()
    return out, (hd, Wd, yd, cwd)


W0 = wl.TINY
CASES = [
    ("tiny", W0, 0),
    # three token chunks of 512 rows, the last one ragged; per-token gradients
    ("ragged_none_chunks", dataclasses.replace(W0, name="f1", N=1100, H=200, V=1000,
                                               reduction="none", grad_mode="normal"), 512),
    # mean over chunks: the denominator counts every chunk's rows
    ("ragged_mean_zloss_chunks", dataclasses.replace(W0, name="f2", N=1300, H=200, V=1000,
                                                     zloss_coef=1e-3), 512),
    ("sum_zloss", dataclasses.replace(W0, name="f3", N=260, H=128, V=776, reduction="sum",
                                      zloss_coef=1e-2, ignore_frac=0.2), 0),
    ("softcap_tight_chunks", dataclasses.replace(W0, name="f4", N=1124, H=256, V=2048,
                                                 w_std=0.3, softcap=2.0, reduction="none",
                                                 grad_mode="normal"), 512),
    ("softcap_30", dataclasses.replace(W0, name="f5", N=256, H=576, V=2992, w_std=0.03,
                                       softcap=30.0), 0),
    ("rl_self_labels", dataclasses.replace(W0, name="f6", N=512, H=448, V=2048,
                                           reduction="none", label_mode="self", grad_mode="rl",
                                           ignore_frac=0.15), 0),
    ("one_row", dataclasses.replace(W0, name="f7", N=1, H=8, V=8, ignore_frac=0.0), 0),
]
LAYOUT_CASES = [c for c in CASES if c[0] in ("ragged_none_chunks", "softcap_30", "tiny")] + [
    # a [V,H] weight takes any vocabulary size (not a multiple of 8 here)
    ("odd_vocab_chunks", dataclasses.replace(W0, name="f8", N=1100, H=200, V=1001,
                                             reduction="none", grad_mode="normal"), 512),
    ("odd_vocab_mean_cap", dataclasses.replace(W0, name="f9", N=300, H=128, V=2003, w_std=0.2,
                                               softcap=4.0, zloss_coef=1e-3), 0),
]


def check_against_oracle(w, chunk_n, layout="hv", eps=0.0, cw=None):
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    h = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    y = labels.numpy()
    okw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, label_smoothing=eps,
               class_weight=None if cw is None else cw.numpy())
    o = orc.forward(h, W, y, w.reduction, **okw)
    dh_o, dw_o = orc.backward(h, W, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                              w.reduction, **okw)
    (loss, ent, lse, ez, dh, dw), _ = run_fused(w, hidden, weight, labels, g_loss, g_ent,
                                                chunk_n, layout, eps, cw)
    if layout == "vh":
        assert dw.shape == (w.V, w.H)
        dw = dw.t()
    valid = o["valid"]
    assert np.abs(f64(lse) - o["lse"]).max() <= TOK_ABS
    assert np.abs(f64(ez) - o["ez"]).max() <= TOK_ABS
    if w.reduction == "none":
        assert np.abs(f64(loss) - o["loss"]).max() <= TOK_ABS
        assert np.abs(f64(ent) - o["entropy"]).max() <= TOK_ABS
        assert np.all(f64(loss)[~valid] == 0) and np.all(f64(ent)[~valid] == 0)
    else:
        for got, ref in ((float(loss[0]), float(o["loss"])), (float(ent[0]), float(o["entropy"]))):
            assert abs(got - ref) <= RED_REL * abs(ref) if ref != 0 else got == 0
    e_dh, e_dw = rel_l2(f64(dh), dh_o), rel_l2(f64(dw), dw_o)
    assert e_dh <= GRAD_REL_L2, e_dh
    assert e_dw <= GRAD_REL_L2, e_dw
    ign = np.nonzero(~valid)[0]
    if ign.size:
        assert torch.all(dh.cpu()[torch.from_numpy(ign)].view(torch.int16) == 0)


@pytest.mark.parametrize("name,w,chunk_n", CASES, ids=[c[0] for c in CASES])
def test_fused_parity(name, w, chunk_n):
    _cuda_or_skip()
    check_against_oracle(w, chunk_n)


@pytest.mark.parametrize("name,w,chunk_n", LAYOUT_CASES, ids=[c[0] for c in LAYOUT_CASES])
def test_fused_parity_vh_layout(name, w, chunk_n):
    _cuda_or_skip()
    check_against_oracle(w, chunk_n, layout="vh")


def test_fused_label_smoothing_and_class_weights_chunked():
    _cuda_or_skip()
    w = dataclasses.replace(W0, name="f8", N=1100, H=192, V=1000, zloss_coef=1e-3)
    g = torch.Generator().manual_seed(7)
    cw = (torch.rand(w.V, generator=g) * 1.5 + 0.25).float()
    check_against_oracle(w, 512, eps=0.1, cw=cw)
    check_against_oracle(dataclasses.replace(w, reduction="none", grad_mode="normal"), 512,
                         layout="vh", eps=0.05)


@pytest.mark.parametrize("name,w,chunk_n", CASES[:6], ids=[c[0] for c in CASES[:6]])
@pytest.mark.parametrize("layout", ["hv", "vh"])
def test_fused_agrees_with_two_call_path(name, w, chunk_n, layout):
    """Forward outputs bitwise equal; dweight bitwise equal with one token chunk."""
    _cuda_or_skip()
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    (loss, ent, lse, ez, dh, dw), (hd, Wd, yd, _) = run_fused(
        w, hidden, weight, labels, g_loss, g_ent, chunk_n, layout)
    kw = _kw(w, layout, 0.0, None)
    loss2, ent2, lse2, ez2 = flce_forward(hd, Wd, yd, w.reduction, validate=True, **kw)
    dh2, dw2 = flce_backward(hd, Wd, yd, lse2, ez2, g_loss.cuda(), g_ent.cuda(), w.reduction,
                             validate=True, **kw)
    torch.cuda.synchronize()
    for a, b in ((lse, lse2), (ez, ez2), (loss, loss2), (ent, ent2)):
        assert torch.equal(a, b)
    one_chunk = chunk_n == 0 or w.N <= chunk_n
    if one_chunk:
        assert torch.equal(dw.view(torch.int16), dw2.view(torch.int16))
    else:
        assert rel_l2(f64(dw), f64(dw2)) <= 4e-3
    # dhidden sums all of V in one contraction (the two-call path: fp32 over chunks)
    assert rel_l2(f64(dh), f64(dh2)) <= 4e-3


def test_fused_empty_batch_zeroes_dweight():
    _cuda_or_skip()
    dev = torch.device("cuda")
    hd = torch.zeros(0, 64, dtype=torch.bfloat16, device=dev)
    Wd = torch.randn(64, 256, device=dev).to(torch.bfloat16)
    yd = torch.zeros(0, dtype=torch.int64, device=dev)
    one = torch.ones(1, device=dev)
    loss, ent, lse, ez, dh, dw = flce_forward_backward(hd, Wd, yd, one, one, "mean",
                                                       validate=True)
    torch.cuda.synchronize()
    assert float(loss[0]) == 0.0 and float(ent[0]) == 0.0
    assert torch.all(dw.view(torch.int16) == 0)


def test_fused_bad_label_reported():
    _cuda_or_skip()
    from linear_cross_entropy_forward_gb300 import FlceError
    dev = torch.device("cuda")
    hd = torch.randn(64, 64, device=dev).to(torch.bfloat16)
    Wd = torch.randn(64, 256, device=dev).to(torch.bfloat16)
    yd = torch.zeros(64, dtype=torch.int64, device=dev)
    yd[5] = 999
    one = torch.ones(1, device=dev)
    with pytest.raises(FlceError, match="LABEL"):
        flce_forward_backward(hd, Wd, yd, one, one, "mean", validate=True)


@pytest.mark.parametrize("n", [8, 1003, 1 << 20])
def test_scale_bf16_matches_rounded_product(n):
    _cuda_or_skip()
    dev = torch.device("cuda")
    x = torch.randn(n, device=dev).to(torch.bfloat16)
    ref = (x.float() * 0.37).to(torch.bfloat16)
    y = x.clone()
    flce_scale_bf16(y, torch.tensor([0.37], device=dev))
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    z = x.clone()
    flce_scale_bf16(z, torch.ones(1, device=dev))
    assert torch.equal(z.view(torch.int16), x.view(torch.int16))
    # a negative scale: the product rounded the same way, zeros kept as +0
    x[::3] = 0.0
    ref = (x.float() * -0.37).to(torch.bfloat16)
    ref[ref == 0] = 0.0
    y = x.clone()
    flce_scale_bf16(y, torch.tensor([-0.37], device=dev))
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert torch.all(y[::3].view(torch.int16) == 0)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_autograd_grad_in_forward(reduction):
    """loss + c * entropy through the grad-in-forward autograd mode against the
    two-call autograd path, with an upstream gradient of 2 (bf16-exact scaling)."""
    _cuda_or_skip()
    w = dataclasses.replace(W0, name="f9", N=700, H=256, V=1536, zloss_coef=1e-3,
                            reduction=reduction)
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    dev = torch.device("cuda")
    c = -0.25
    grads = []
    for gif in (False, True):
        h = hidden.to(dev).requires_grad_(True)
        W = weight.to(dev).requires_grad_(True)
        loss, ent = linear_cross_entropy(h, W, labels.to(dev), reduction,
                                         zloss_coef=w.zloss_coef, grad_in_forward=gif,
                                         entropy_coef=c)
        obj = 2.0 * loss if gif else 2.0 * (loss + c * ent)
        obj.backward()
        grads.append((float(loss.detach()), float(ent.detach()), h.grad.clone(), W.grad.clone()))
    (l0, e0, dh0, dw0), (l1, e1, dh1, dw1) = grads
    assert l0 == l1 and e0 == e1
    assert rel_l2(f64(dh1), f64(dh0)) <= 4e-3
    assert rel_l2(f64(dw1), f64(dw0)) <= 4e-3


def test_autograd_grad_in_forward_rejects_none_reduction():
    _cuda_or_skip()
    dev = torch.device("cuda")
    h = torch.randn(64, 64, device=dev).to(torch.bfloat16).requires_grad_(True)
    W = torch.randn(64, 256, device=dev).to(torch.bfloat16).requires_grad_(True)
    y = torch.zeros(64, dtype=torch.int64, device=dev)
    with pytest.raises(ValueError):
        linear_cross_entropy(h, W, y, "none", grad_in_forward=True)


FULL = [wl.LLAMA3, wl.QWEN25]


@pytest.mark.slow
@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_fused_fullsize_against_two_call_and_oracle_rows(w):
    """Bench-size workloads with the default token chunk (Llama-3 head: one chunk;
    Qwen2.5 RL batch: two, with fp32 dweight accumulation): forward outputs bitwise
    equal to the two-call path, gradients close to it; every row's lse and E_p[z],
    sampled dhidden rows and sampled dweight columns against the oracle."""
    _cuda_or_skip()
    dev = torch.device("cuda")
    label_dev = "cuda" if w.label_mode == "self" else "cpu"
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w, label_device=label_dev)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    gl, ge = g_loss.to(dev), g_ent.to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)
    loss, ent, lse, ez, dh, dw = flce_forward_backward(hd, Wd, yd, gl, ge, w.reduction,
                                                       validate=True, **kw)
    loss2, ent2, lse2, ez2 = flce_forward(hd, Wd, yd, w.reduction, validate=True, **kw)
    for a, b in ((lse, lse2), (ez, ez2), (loss, loss2), (ent, ent2)):
        assert torch.equal(a, b)
    del loss2, ent2
    dh2, dw2 = flce_backward(hd, Wd, yd, lse2, ez2, gl, ge, w.reduction, validate=True, **kw)
    torch.cuda.synchronize()
    assert torch.isfinite(dh.float()).all() and torch.isfinite(dw.float()).all()
    assert float((dh.float() - dh2.float()).norm() / dh2.float().norm()) <= 4e-3
    assert float((dw.float() - dw2.float()).norm() / dw2.float().norm()) <= 4e-3
    del dh2, dw2
    # every row's forward outputs against the oracle (row statistics cached per process)
    hb, wb = wl.bf16_bits(hidden), wl.bf16_bits(weight)
    h64 = orc.bf16_bits_to_f64(hb)
    W64 = orc.bf16_bits_to_f64(wb)
    y = labels.cpu().numpy()
    st = fso.row_stats(hb, wb, h64, W64, w.softcap)
    o = orc.forward(h64, W64, y, "none", stats=st, **kw)
    assert np.abs(f64(lse) - o["lse"]).max() <= TOK_ABS
    assert np.abs(f64(ez) - o["ez"]).max() <= TOK_ABS
    # dhidden on sampled rows, dweight on sampled columns (with several token chunks the
    # columns hold the fp32 accumulation across chunks)
    rng = np.random.default_rng(99)
    rows = np.unique(np.concatenate([rng.choice(w.N, 24, replace=False), [0, w.N - 1]]))
    dh_o, _ = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                           w.reduction, rows=rows, **kw)
    assert rel_l2(f64(dh[torch.from_numpy(rows).to(dev)]), dh_o) <= GRAD_REL_L2
    cols = fso.dweight_columns(w.V, y)
    _, dw_o = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                           w.reduction, cols=cols, **kw)
    assert rel_l2(f64(dw[:, torch.from_numpy(cols).to(dev)]), dw_o) <= GRAD_REL_L2
