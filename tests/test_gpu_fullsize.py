"""Full-size parity in the launch configuration bench.py times (default chunking).

Every row's lse / E_p[z] / loss / entropy and the reduced outputs are compared with
the fp64 oracle over the whole batch (its row statistics are computed once per
process and cached, see _fullsize_oracle.py).  dhidden is compared on seeded row
samples (each row needs only its own row of logits) and dweight on at least 64
sampled vocabulary columns (each column needs only its own column of logits and
every row's statistics): label columns, columns in every backward vocabulary chunk,
and the last, ragged vocabulary tile.  The Llama-2 head shape is also compared
element by element against the complete oracle.
"""
import numpy as np
import pytest
import torch

import _fullsize_oracle as fso
from linear_cross_entropy_forward_gb300 import (flce_backward, flce_forward,
                                                flce_forward_backward)
from linear_cross_entropy_forward_gb300 import workloads as wl
from oracle import flce_oracle as orc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOK_ABS = 2e-3
RED_REL = 1e-4
GRAD_REL_L2 = 1e-2
N_SAMPLE = 48

FULL = [wl.LLAMA2, wl.LLAMA3, wl.GEMMA2, wl.QWEN25]


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    build()


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def sample_rows(w, labels):
    rng = np.random.default_rng(1234)
    y = labels.numpy()
    ign = np.nonzero(y == wl.IGNORE_INDEX)[0]
    val = np.nonzero(y != wl.IGNORE_INDEX)[0]
    pick = list(rng.choice(val, size=N_SAMPLE - 4, replace=False))
    if ign.size:
        pick += list(rng.choice(ign, size=min(4, ign.size), replace=False))
    # the first and last rows exercise the edge tiles
    pick += [0, w.N - 1]
    return np.unique(np.array(pick, dtype=np.int64))


def oracle_whole_batch(w, hidden, weight, labels, reduction, **kw):
    """The oracle's forward over every row (row statistics from the cache), plus the
    fp64 inputs it used."""
    hb, wb = wl.bf16_bits(hidden), wl.bf16_bits(weight)
    h64 = orc.bf16_bits_to_f64(hb)
    W64 = orc.bf16_bits_to_f64(wb)
    st = fso.row_stats(hb, wb, h64, W64, kw.get("softcap", 0.0))
    o = orc.forward(h64, W64, labels.cpu().numpy(), reduction, stats=st, **kw)
    return o, h64, W64, st


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_fullsize_parity(w):
    _cuda_or_skip()
    dev = torch.device("cuda")
    label_dev = "cuda" if w.label_mode == "self" else "cpu"
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w, label_device=label_dev)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)
    loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, validate=True, **kw)
    dh, dw = flce_backward(hd, Wd, yd, lse, ez, g_loss.to(dev), g_ent.to(dev), w.reduction,
                           validate=True, **kw)
    if w.reduction != "none":
        loss_t, ent_t, _, _ = flce_forward(hd, Wd, yd, "none", validate=True, **kw)
    else:
        loss_t, ent_t = loss, ent
    torch.cuda.synchronize()
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    g_lse, g_ez, g_lt, g_et = f64(lse), f64(ez), f64(loss_t), f64(ent_t)
    valid = labels.numpy() != wl.IGNORE_INDEX
    assert np.all(g_lt[~valid] == 0) and np.all(g_et[~valid] == 0)

    # every row against the oracle
    o, h64, W64, st = oracle_whole_batch(w, hidden, weight, labels, "none", **kw)
    assert np.abs(g_lse - o["lse"]).max() <= TOK_ABS
    assert np.abs(g_ez - o["ez"]).max() <= TOK_ABS
    assert np.abs(g_lt - o["loss_tok"]).max() <= TOK_ABS
    assert np.abs(g_et - o["entropy_tok"]).max() <= TOK_ABS
    if w.reduction != "none":
        o_red = orc.forward(h64, W64, labels.numpy(), w.reduction, stats=st, **kw)
        assert abs(float(loss.item()) - o_red["loss"]) <= RED_REL * abs(o_red["loss"])
        assert abs(float(ent.item()) - o_red["entropy"]) <= RED_REL * abs(o_red["entropy"])

    # dhidden on sampled rows (each needs its own row of logits)
    y = labels.numpy()
    rows = sample_rows(w, labels)
    dh_o, _ = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                           w.reduction, rows=rows, **kw)
    dh_rows = f64(dh[torch.from_numpy(rows).to(dev)])
    assert rel_l2(dh_rows, dh_o) <= GRAD_REL_L2
    # every ignored row of dhidden is exactly zero
    ign = torch.from_numpy(np.nonzero(~valid)[0]).to(dev)
    if ign.numel():
        assert torch.all(dh[ign].view(torch.int16) == 0)

    # dweight on sampled columns, element by element (each needs its own column of
    # logits and every row's statistics)
    cols = fso.dweight_columns(w.V, y)
    assert cols.size >= 64
    _, dw_o = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                           w.reduction, cols=cols, **kw)
    dw_cols = f64(dw[:, torch.from_numpy(cols).to(dev)])
    assert rel_l2(dw_cols, dw_o) <= GRAD_REL_L2
    # and finite everywhere
    assert torch.isfinite(dw.float()).all()


def test_llama2_head_against_complete_oracle():
    """Llama-2-7B head shape: every output element against the full fp64 oracle."""
    _cuda_or_skip()
    w = wl.LLAMA2
    dev = torch.device("cuda")
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, validate=True)
    dh, dw = flce_backward(hd, Wd, yd, lse, ez, g_loss.to(dev), g_ent.to(dev), w.reduction,
                           validate=True)
    torch.cuda.synchronize()
    h64 = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W64 = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    y = labels.numpy()
    o = orc.forward(h64, W64, y, w.reduction)
    dh_o, dw_o = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(),
                              w.reduction)
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    assert np.abs(f64(loss) - o["loss"]).max() <= TOK_ABS
    assert np.abs(f64(ent) - o["entropy"]).max() <= TOK_ABS
    assert np.abs(f64(lse) - o["lse"]).max() <= TOK_ABS
    assert rel_l2(f64(dh), dh_o) <= GRAD_REL_L2
    assert rel_l2(f64(dw), dw_o) <= GRAD_REL_L2


def test_fullsize_weight_layouts_agree_bitwise():
    """Gemma-2 head shape (soft-cap 30, V = 256000): the nn.Linear layout [V,H] gives the
    same bits as [H,V] for every output (the layouts change operand majorness and tile
    order, never the order of any element's accumulation)."""
    _cuda_or_skip()
    w = wl.GEMMA2
    dev = torch.device("cuda")
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    hd, yd, gl, ge = hidden.to(dev), labels.to(dev), g_loss.to(dev), g_ent.to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)
    res = {}
    for layout in ("hv", "vh"):
        Wd = weight.to(dev) if layout == "hv" else weight.t().contiguous().to(dev)
        loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, validate=True,
                                          weight_layout=layout, **kw)
        dh, dw = flce_backward(hd, Wd, yd, lse, ez, gl, ge, w.reduction, validate=True,
                               weight_layout=layout, **kw)
        torch.cuda.synchronize()
        res[layout] = (loss, ent, lse, ez, dh, (dw if layout == "hv" else dw.t()).contiguous())
        del Wd
    for a, b in zip(res["hv"], res["vh"]):
        if a.dtype == torch.bfloat16:
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        else:
            assert torch.equal(a, b)


def test_qwen_batch_with_arrays_past_2_31_elements():
    """Qwen2.5 RL batch (N = 16384, V = 152064) with the whole problem in one chunk: the
    backward's dlogits chunk of all 152064 columns and the gradient-in-forward call's kept
    logits of all 16384 rows each hold 2.49e9 elements (5.0 and 10.0 GB), more than 2^31,
    so the epilogue stores, the TMA maps over these arrays and dlogits_from_z all index
    past it.  dweight does not depend on the vocabulary chunking (every column sums over
    the rows in the same order): bitwise that of the default chunks.  The two one-chunk
    runs form the same dlogits and contract them the same way, so they agree bit for bit.
    dhidden rows and dweight columns against the oracle."""
    _cuda_or_skip()
    w = wl.QWEN25
    assert w.N * w.V > 2 ** 31 and w.V % 256 == 0 and w.N % 512 == 0
    dev = torch.device("cuda")
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w, label_device="cuda")
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    gl, ge = g_loss.to(dev), g_ent.to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap)
    loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, validate=True, **kw)
    _, dw_d = flce_backward(hd, Wd, yd, lse, ez, gl, ge, w.reduction, validate=True, **kw)
    dh_1, dw_1 = flce_backward(hd, Wd, yd, lse, ez, gl, ge, w.reduction, validate=True,
                               chunk_v=w.V, **kw)
    torch.cuda.synchronize()
    assert torch.equal(dw_1.view(torch.int16), dw_d.view(torch.int16))
    del dw_d
    torch.cuda.empty_cache()
    out = flce_forward_backward(hd, Wd, yd, gl, ge, w.reduction, validate=True, chunk_n=w.N,
                                **kw)
    torch.cuda.synchronize()
    for a, b in zip(out[:4], (loss, ent, lse, ez)):
        assert torch.equal(a, b)
    assert torch.equal(out[4].view(torch.int16), dh_1.view(torch.int16))
    assert torch.equal(out[5].view(torch.int16), dw_1.view(torch.int16))
    del out
    torch.cuda.empty_cache()

    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    o, h64, W64, _ = oracle_whole_batch(w, hidden, weight, labels, "none", **kw)
    assert np.abs(f64(lse) - o["lse"]).max() <= TOK_ABS
    y = labels.cpu().numpy()
    rows = sample_rows(w, labels.cpu())
    dh_o, _ = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.cpu().numpy(),
                           g_ent.cpu().numpy(), w.reduction, rows=rows, **kw)
    assert rel_l2(f64(dh_1[torch.from_numpy(rows).to(dev)]), dh_o) <= GRAD_REL_L2
    cols = fso.dweight_columns(w.V, y)
    _, dw_o = orc.backward(h64, W64, y, o["lse"], o["ez"], g_loss.cpu().numpy(),
                           g_ent.cpu().numpy(), w.reduction, cols=cols, **kw)
    assert rel_l2(f64(dw_1[:, torch.from_numpy(cols).to(dev)]), dw_o) <= GRAD_REL_L2
