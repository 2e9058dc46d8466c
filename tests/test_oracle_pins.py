"""Pins for the fp64 oracle: it is checked against things other than itself.

Closed forms, invariants, finite differences, textbook library routines and a
scalar-loop brute force, chosen so that a dropped term, a wrong sign, a wrong
index or a transposed operand in the oracle fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import flce_oracle as orc
from oracle import loop_checker as lc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
REDS = ("none", "mean", "sum")


def _rand_case(N, H, V, seed, w_std=0.5, ignore=(1,)):
    rng = np.random.default_rng(seed)
    hidden = rng.standard_normal((N, H))
    weight = rng.standard_normal((H, V)) * w_std
    labels = rng.integers(0, V, N)
    for i in ignore:
        if i < N:
            labels[i] = orc.IGNORE_INDEX
    return hidden, weight, labels


def _grads(reduction, N, seed):
    rng = np.random.default_rng(seed + 100)
    if reduction == "none":
        return rng.standard_normal(N), rng.standard_normal(N)
    return np.array([0.7]), np.array([-1.3])


# --------------------------------------------------------------------------- bf16
def test_bf16_widening_is_exact_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


# --------------------------------------------------------------------------- worked examples
def _ev(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, vars(math)))
    return float(x)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_worked_examples(case):
    hidden = np.array([[_ev(x) for x in r] for r in case["hidden"]])
    weight = np.array([[_ev(x) for x in r] for r in case["weight"]])
    labels = np.array(case["labels"])
    out = orc.forward(hidden, weight, labels, "none", zloss_coef=case["zloss_coef"],
                      softcap=case["softcap"])
    np.testing.assert_allclose(out["lse"], [_ev(x) for x in case["lse"]], rtol=0, atol=1e-13)
    np.testing.assert_allclose(out["ce_tok"], [_ev(x) for x in case["ce"]], rtol=0, atol=1e-13)
    np.testing.assert_allclose(out["entropy_tok"], [_ev(x) for x in case["entropy"]], rtol=0,
                               atol=1e-13)
    if "loss" in case:
        np.testing.assert_allclose(out["loss_tok"], [_ev(x) for x in case["loss"]], rtol=0,
                                   atol=1e-13)
    if "backward" in case:
        b = case["backward"]
        dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"],
                              np.array(b["g_loss"]), np.array(b["g_entropy"]), "none",
                              zloss_coef=case["zloss_coef"], softcap=case["softcap"])
        np.testing.assert_allclose(dw, [[_ev(x) for x in r] for r in b["dweight"]], rtol=0,
                                   atol=1e-13)
        np.testing.assert_allclose(dh, [[_ev(x) for x in r] for r in b["dhidden"]], rtol=0,
                                   atol=1e-13)


# --------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("reduction", REDS)
@pytest.mark.parametrize("zc", [0.0, 0.05])
@pytest.mark.parametrize("cap", [0.0, 5.0])
def test_zero_weight_closed_form(reduction, zc, cap):
    """weight = 0: every logit is 0, p is uniform, CE = entropy = lse = ln V; the
    entropy gradient vanishes; dhidden = 0 and dweight[:, v] = sum_n g_n h_n (1/V - [y_n = v])
    plus the z-loss term 2 coef ln V / V sum_n g_n h_n."""
    N, H, V = 9, 6, 11
    rng = np.random.default_rng(3)
    hidden = rng.standard_normal((N, H))
    weight = np.zeros((H, V))
    labels = rng.integers(0, V, N)
    labels[[2, 5]] = orc.IGNORE_INDEX
    valid = labels != orc.IGNORE_INDEX
    out = orc.forward(hidden, weight, labels, reduction, zloss_coef=zc, softcap=cap)
    lnv = math.log(V)
    np.testing.assert_allclose(out["lse"], lnv, atol=1e-14)
    np.testing.assert_allclose(out["ce_tok"][valid], lnv, atol=1e-14)
    np.testing.assert_allclose(out["entropy_tok"][valid], lnv, atol=1e-14)
    assert np.all(out["ce_tok"][~valid] == 0) and np.all(out["entropy_tok"][~valid] == 0)
    gl_in, ge_in = _grads(reduction, N, 3)
    dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl_in, ge_in,
                          reduction, zloss_coef=zc, softcap=cap)
    assert np.max(np.abs(dh)) < 1e-14
    # upstream grads after the reduction (independent restatement of the scaling rule)
    g = np.broadcast_to(gl_in, (N,)).astype(float).copy()
    if reduction == "mean":
        g /= valid.sum()
    g[~valid] = 0
    expect = np.zeros((H, V))
    for n in range(N):
        for v in range(V):
            expect[:, v] += g[n] * hidden[n] * (1.0 / V - (labels[n] == v) + 2 * zc * lnv / V)
    np.testing.assert_allclose(dw, expect, atol=1e-13)


@pytest.mark.parametrize("zc", [0.0, 0.1])
def test_single_class(zc):
    """V = 1: p = 1, CE = 0, entropy = 0, lse = z and the loss is coef * z^2."""
    rng = np.random.default_rng(4)
    hidden = rng.standard_normal((5, 3))
    weight = rng.standard_normal((3, 1))
    labels = np.zeros(5, dtype=np.int64)
    out = orc.forward(hidden, weight, labels, "none", zloss_coef=zc)
    z = (hidden @ weight)[:, 0]
    np.testing.assert_allclose(out["ce_tok"], 0.0, atol=1e-14)
    np.testing.assert_allclose(out["entropy_tok"], 0.0, atol=1e-14)
    np.testing.assert_allclose(out["loss_tok"], zc * z * z, atol=1e-13)


def test_all_ignored_mean_is_zero():
    hidden, weight, _ = _rand_case(4, 3, 5, 5)
    labels = np.full(4, orc.IGNORE_INDEX)
    out = orc.forward(hidden, weight, labels, "mean")
    assert out["loss"] == 0.0 and out["entropy"] == 0.0 and out["n_valid"] == 0
    dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], [1.0], [1.0], "mean")
    assert not dh.any() and not dw.any()


# --------------------------------------------------------------------------- textbook routines
@pytest.mark.parametrize("reduction", REDS)
def test_matches_torch_cross_entropy_and_logsumexp(reduction):
    """No soft-cap, no z-loss: the loss is torch's cross_entropy (float64, ignore_index=-100),
    lse is torch.logsumexp and the entropy is scipy's Shannon entropy of the softmax."""
    from scipy.stats import entropy as shannon
    hidden, weight, labels = _rand_case(37, 19, 301, 6, w_std=0.8, ignore=(0, 5, 9))
    out = orc.forward(hidden, weight, labels, reduction, v_chunk=64)
    z = torch.from_numpy(hidden) @ torch.from_numpy(weight)
    y = torch.from_numpy(labels)
    ref = torch.nn.functional.cross_entropy(z, y, ignore_index=-100, reduction=reduction)
    np.testing.assert_allclose(out["loss"], ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["lse"], torch.logsumexp(z, dim=1).numpy(), rtol=1e-13)
    p = torch.softmax(z, dim=1).numpy()
    valid = labels != orc.IGNORE_INDEX
    ent = np.where(valid, shannon(p, axis=1), 0.0)
    if reduction == "none":
        np.testing.assert_allclose(out["entropy"], ent, rtol=1e-11, atol=1e-12)
    elif reduction == "sum":
        np.testing.assert_allclose(out["entropy"], ent.sum(), rtol=1e-11)
    else:
        np.testing.assert_allclose(out["entropy"], ent.sum() / valid.sum(), rtol=1e-11)


def test_zloss_adds_coef_lse_squared():
    hidden, weight, labels = _rand_case(11, 7, 50, 7, ignore=(3,))
    a = orc.forward(hidden, weight, labels, "sum", zloss_coef=0.0)
    b = orc.forward(hidden, weight, labels, "sum", zloss_coef=0.01)
    z = torch.from_numpy(hidden) @ torch.from_numpy(weight)
    lse = torch.logsumexp(z, dim=1).numpy()
    valid = labels != orc.IGNORE_INDEX
    np.testing.assert_allclose(b["loss"] - a["loss"], 0.01 * (lse[valid] ** 2).sum(), rtol=1e-12)
    assert b["entropy"] == a["entropy"]


# --------------------------------------------------------------------------- invariants
@pytest.mark.parametrize("cap", [0.0, 2.0])
def test_entropy_and_ce_bounds(cap):
    hidden, weight, labels = _rand_case(64, 16, 97, 8, w_std=2.0, ignore=())
    out = orc.forward(hidden, weight, labels, "none", softcap=cap, v_chunk=32)
    assert np.all(out["entropy_tok"] >= -1e-12)
    assert np.all(out["entropy_tok"] <= math.log(97) + 1e-12)
    assert np.all(out["ce_tok"] >= -1e-12)


def test_softcap_bounds_and_large_cap_limit():
    hidden, weight, labels = _rand_case(16, 8, 40, 9, w_std=5.0)
    z = orc.logits_chunk(hidden, weight, 0, 40, softcap=3.0)
    # tanh rounds to exactly 1 for large arguments in fp64, so the bound is closed
    assert np.all(np.abs(z) <= 3.0)
    zp = hidden @ weight
    moderate = np.abs(zp) < 30.0
    assert np.all(np.abs(z[moderate]) < 3.0)
    assert np.all(np.sign(z) == np.sign(zp))
    a = orc.forward(hidden, weight, labels, "none", softcap=0.0)
    b = orc.forward(hidden, weight, labels, "none", softcap=1e7)
    np.testing.assert_allclose(b["loss"], a["loss"], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(b["entropy"], a["entropy"], rtol=1e-9, atol=1e-9)


def test_chunking_does_not_change_results():
    hidden, weight, labels = _rand_case(20, 9, 103, 10)
    for cap in (0.0, 4.0):
        a = orc.forward(hidden, weight, labels, "none", softcap=cap, zloss_coef=0.01, v_chunk=7)
        b = orc.forward(hidden, weight, labels, "none", softcap=cap, zloss_coef=0.01, v_chunk=4096)
        np.testing.assert_allclose(a["loss"], b["loss"], rtol=1e-13)
        np.testing.assert_allclose(a["ez"], b["ez"], rtol=1e-12, atol=1e-13)
        gl, ge = _grads("none", 20, 10)
        da = orc.backward(hidden, weight, labels, a["lse"], a["ez"], gl, ge, "none",
                          softcap=cap, zloss_coef=0.01, v_chunk=7)
        db = orc.backward(hidden, weight, labels, b["lse"], b["ez"], gl, ge, "none",
                          softcap=cap, zloss_coef=0.01, v_chunk=4096)
        np.testing.assert_allclose(da[0], db[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(da[1], db[1], rtol=1e-12, atol=1e-14)


def test_shift_invariance():
    """A constant added to every logit of a row (a constant feature times a constant
    weight row) changes neither CE, entropy nor dhidden of the original features."""
    hidden, weight, labels = _rand_case(12, 6, 33, 11)
    h2 = np.concatenate([hidden, np.ones((12, 1))], axis=1)
    w2 = np.concatenate([weight, np.full((1, 33), 4.25)], axis=0)
    a = orc.forward(hidden, weight, labels, "none")
    b = orc.forward(h2, w2, labels, "none")
    np.testing.assert_allclose(b["ce_tok"], a["ce_tok"], atol=1e-12)
    np.testing.assert_allclose(b["entropy_tok"], a["entropy_tok"], atol=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"] + 4.25, atol=1e-12)
    gl, ge = _grads("none", 12, 11)
    da, _ = orc.backward(hidden, weight, labels, a["lse"], a["ez"], gl, ge, "none")
    db, _ = orc.backward(h2, w2, labels, b["lse"], b["ez"], gl, ge, "none")
    np.testing.assert_allclose(db[:, :6], da, atol=1e-12)


@pytest.mark.parametrize("cap", [0.0, 3.0])
def test_dlogit_rows_sum(cap):
    """sum_v (p - onehot) = 0 and sum_v p (z - E_p z) = 0, so without z-loss (and without the
    cap's chain term) every dlogits row sums to 0; with z-loss it sums to 2 coef lse g."""
    hidden, weight, labels = _rand_case(15, 7, 64, 12)
    for zc in (0.0, 0.02):
        out = orc.forward(hidden, weight, labels, "none", zloss_coef=zc)
        gl, ge = _grads("none", 15, 12)
        gcs, gls, ges = orc.grad_scales(gl, ge, out["valid"], "none")
        dz = orc.dlogits_chunk(hidden, weight, labels, out["lse"], out["ez"], gcs, gls, ges, 0,
                               64, zloss_coef=zc)
        np.testing.assert_allclose(dz.sum(axis=1), 2 * zc * out["lse"] * gls, atol=1e-12)
        if cap == 0.0 and zc == 0.0:
            _, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, "none")
            np.testing.assert_allclose(dw.sum(axis=1), 0.0, atol=1e-12)


# --------------------------------------------------------------------------- finite differences
@pytest.mark.parametrize("reduction", REDS)
@pytest.mark.parametrize("zc", [0.0, 0.1])
@pytest.mark.parametrize("cap", [0.0, 1.5])
def test_backward_matches_finite_differences(reduction, zc, cap):
    N, H, V = 6, 5, 9
    hidden, weight, labels = _rand_case(N, H, V, 20, w_std=0.7, ignore=(2,))
    gl, ge = _grads(reduction, N, 20)
    out = orc.forward(hidden, weight, labels, reduction, zloss_coef=zc, softcap=cap)
    dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction,
                          zloss_coef=zc, softcap=cap)
    kw = dict(reduction=reduction, zloss_coef=zc, softcap=cap)
    eps = 1e-6
    fd_h = np.zeros_like(hidden)
    for n in range(N):
        for h in range(H):
            hp, hm = hidden.copy(), hidden.copy()
            hp[n, h] += eps
            hm[n, h] -= eps
            fd_h[n, h] = (orc.objective(hp, weight, labels, gl, ge, **kw)
                          - orc.objective(hm, weight, labels, gl, ge, **kw)) / (2 * eps)
    fd_w = np.zeros_like(weight)
    for h in range(H):
        for v in range(V):
            wp, wm = weight.copy(), weight.copy()
            wp[h, v] += eps
            wm[h, v] -= eps
            fd_w[h, v] = (orc.objective(hidden, wp, labels, gl, ge, **kw)
                          - orc.objective(hidden, wm, labels, gl, ge, **kw)) / (2 * eps)
    scale_h = max(1.0, np.abs(fd_h).max())
    scale_w = max(1.0, np.abs(fd_w).max())
    assert np.abs(dh - fd_h).max() / scale_h < 1e-6
    assert np.abs(dw - fd_w).max() / scale_w < 1e-6
    assert not dh[2].any()  # ignored row


def test_rows_subset_backward_equals_full():
    hidden, weight, labels = _rand_case(10, 4, 30, 21)
    gl, ge = _grads("none", 10, 21)
    out = orc.forward(hidden, weight, labels, "none", zloss_coef=0.01, softcap=2.0)
    dh, _ = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, "none",
                         zloss_coef=0.01, softcap=2.0)
    rows = np.array([7, 1, 4])
    dhr, none = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, "none",
                             zloss_coef=0.01, softcap=2.0, rows=rows, v_chunk=8)
    assert none is None
    np.testing.assert_allclose(dhr, dh[rows], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("reduction", REDS)
@pytest.mark.parametrize("opts", [dict(), dict(zloss_coef=0.01, softcap=2.0),
                                  dict(label_smoothing=0.1, class_weight="random")],
                         ids=["plain", "zloss_softcap", "smooth_weighted"])
def test_column_subset_backward_equals_full(reduction, opts):
    """dweight[:, cols] over every row (the form the full-size GPU checks use) equals the
    columns of the complete dweight, itself pinned by finite differences above."""
    hidden, weight, labels = _rand_case(12, 5, 30, 23, ignore=(2, 9))
    kw = dict(opts)
    if kw.get("class_weight") == "random":
        kw["class_weight"] = np.random.default_rng(5).uniform(0.5, 2.0, 30)
    gl, ge = _grads(reduction, 12, 23)
    out = orc.forward(hidden, weight, labels, reduction, **kw)
    _, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction, **kw)
    cols = np.array([0, int(labels[0]), 29, 17, int(labels[5])])
    none, dwc = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction,
                             cols=cols, **kw)
    assert none is None and dwc.shape == (5, cols.size)
    np.testing.assert_allclose(dwc, dw[:, cols], rtol=1e-12, atol=1e-14)
    with pytest.raises(ValueError):
        orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction,
                     cols=[30], **kw)


def test_column_subset_matches_finite_differences():
    """Each returned dweight column against central differences of the objective in the
    entries of that weight column (soft-cap and z-loss on, mean reduction)."""
    hidden, weight, labels = _rand_case(6, 4, 20, 31)
    kw = dict(zloss_coef=0.05, softcap=1.5)
    gl, ge = np.array([0.8]), np.array([-0.6])
    out = orc.forward(hidden, weight, labels, "mean", **kw)
    cols = np.array([int(labels[0]), 3, 19])
    _, dwc = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, "mean",
                          cols=cols, **kw)
    eps = 1e-6
    fd = np.zeros_like(dwc)
    for i, c in enumerate(cols):
        for h in range(4):
            wp, wm = weight.copy(), weight.copy()
            wp[h, c] += eps
            wm[h, c] -= eps
            fd[h, i] = (orc.objective(hidden, wp, labels, gl, ge, "mean", **kw)
                        - orc.objective(hidden, wm, labels, gl, ge, "mean", **kw)) / (2 * eps)
    assert np.abs(dwc - fd).max() / max(1.0, np.abs(fd).max()) < 1e-6


def test_forward_with_given_row_stats_equals_plain_forward():
    hidden, weight, labels = _rand_case(9, 6, 25, 41)
    cw = np.random.default_rng(6).uniform(0.5, 2.0, 25)
    kw = dict(zloss_coef=0.02, softcap=3.0, label_smoothing=0.05, class_weight=cw)
    plain = orc.forward(hidden, weight, labels, "none", **kw)
    st = orc.row_stats(hidden, weight, 3.0, class_weight=cw)
    given = orc.forward(hidden, weight, labels, "none", stats=st, **kw)
    for k in ("loss", "entropy", "lse", "ez"):
        np.testing.assert_array_equal(np.asarray(given[k]), np.asarray(plain[k]))
    with pytest.raises(ValueError):
        orc.forward(hidden, weight, labels, "none", stats=(st[0][:3], st[1], st[2]), **kw)


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("reduction", REDS)
@pytest.mark.parametrize("zc,cap", [(0.0, 0.0), (0.05, 0.0), (0.0, 2.0), (0.05, 2.0)])
def test_oracle_matches_scalar_loops(reduction, zc, cap):
    N, H, V = 5, 4, 7
    hidden, weight, labels = _rand_case(N, H, V, 30, w_std=0.9, ignore=(1,))
    out = orc.forward(hidden, weight, labels, reduction, zloss_coef=zc, softcap=cap)
    l, e, lse = lc.forward_loops(hidden.tolist(), weight.tolist(), labels.tolist(), reduction,
                                 zloss_coef=zc, softcap=cap)
    np.testing.assert_allclose(out["loss"], l, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out["entropy"], e, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out["lse"], lse, rtol=1e-13)
    gl, ge = _grads(reduction, N, 30)
    dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction,
                          zloss_coef=zc, softcap=cap)
    fh, fw = lc.fd_grads_loops(hidden.tolist(), weight.tolist(), labels.tolist(), gl.tolist(),
                               ge.tolist(), reduction=reduction, zloss_coef=zc, softcap=cap)
    np.testing.assert_allclose(dh, np.array(fh), rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(dw, np.array(fw), rtol=1e-5, atol=1e-7)


# --------------------------------------------------------------------------- smoothing, weights
@pytest.mark.parametrize("reduction", REDS)
@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("weighted", [False, True])
def test_smoothing_and_class_weights_match_torch(reduction, eps, weighted):
    """torch's cross_entropy(weight, label_smoothing, ignore_index) is the definition."""
    hidden, weight, labels = _rand_case(41, 13, 257, 40, w_std=0.9, ignore=(0, 7, 8))
    cw = np.random.default_rng(41).uniform(0.2, 2.0, 257) if weighted else None
    out = orc.forward(hidden, weight, labels, reduction, v_chunk=50, label_smoothing=eps,
                      class_weight=cw)
    z = torch.from_numpy(hidden) @ torch.from_numpy(weight)
    ref = torch.nn.functional.cross_entropy(
        z, torch.from_numpy(labels), weight=None if cw is None else torch.from_numpy(cw),
        ignore_index=-100, reduction=reduction, label_smoothing=eps)
    np.testing.assert_allclose(out["loss"], ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("reduction", REDS)
def test_smoothing_weights_zloss_softcap_finite_differences(reduction):
    N, H, V = 6, 5, 9
    hidden, weight, labels = _rand_case(N, H, V, 50, w_std=0.7, ignore=(2,))
    cw = np.random.default_rng(50).uniform(0.3, 1.7, V)
    gl, ge = _grads(reduction, N, 50)
    kw = dict(zloss_coef=0.05, softcap=2.5, label_smoothing=0.2, class_weight=cw)
    out = orc.forward(hidden, weight, labels, reduction, **kw)
    dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction, **kw)
    eps = 1e-6
    fd_h = np.zeros_like(hidden)
    for n in range(N):
        for h in range(H):
            hp, hm = hidden.copy(), hidden.copy()
            hp[n, h] += eps
            hm[n, h] -= eps
            fd_h[n, h] = (orc.objective(hp, weight, labels, gl, ge, reduction, **kw)
                          - orc.objective(hm, weight, labels, gl, ge, reduction, **kw)) / (2 * eps)
    fd_w = np.zeros_like(weight)
    for h in range(H):
        for v in range(V):
            wp, wm = weight.copy(), weight.copy()
            wp[h, v] += eps
            wm[h, v] -= eps
            fd_w[h, v] = (orc.objective(hidden, wp, labels, gl, ge, reduction, **kw)
                          - orc.objective(hidden, wm, labels, gl, ge, reduction, **kw)) / (2 * eps)
    assert np.abs(dh - fd_h).max() / max(1.0, np.abs(fd_h).max()) < 1e-6
    assert np.abs(dw - fd_w).max() / max(1.0, np.abs(fd_w).max()) < 1e-6


@pytest.mark.parametrize("reduction", REDS)
def test_smoothing_weights_match_scalar_loops(reduction):
    N, H, V = 5, 4, 7
    hidden, weight, labels = _rand_case(N, H, V, 60, w_std=0.9, ignore=(1,))
    cw = np.random.default_rng(60).uniform(0.3, 1.7, V)
    kw = dict(zloss_coef=0.03, softcap=2.0, label_smoothing=0.15, class_weight=cw)
    out = orc.forward(hidden, weight, labels, reduction, **kw)
    l, e, _ = lc.forward_loops(hidden.tolist(), weight.tolist(), labels.tolist(), reduction,
                               zloss_coef=0.03, softcap=2.0, label_smoothing=0.15,
                               class_weight=cw.tolist())
    np.testing.assert_allclose(out["loss"], l, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out["entropy"], e, rtol=1e-12, atol=1e-13)


def test_uniform_class_weights_scale_out_of_the_mean():
    """Scaling every class weight by a constant leaves the mean loss unchanged
    (numerator and denominator scale together) and scales the sum."""
    hidden, weight, labels = _rand_case(20, 6, 30, 70, ignore=(4,))
    a = orc.forward(hidden, weight, labels, "mean", label_smoothing=0.1)
    b = orc.forward(hidden, weight, labels, "mean", label_smoothing=0.1,
                    class_weight=np.full(30, 3.0))
    np.testing.assert_allclose(b["loss"], a["loss"], rtol=1e-12)
    c = orc.forward(hidden, weight, labels, "sum", label_smoothing=0.1)
    d = orc.forward(hidden, weight, labels, "sum", label_smoothing=0.1,
                    class_weight=np.full(30, 3.0))
    np.testing.assert_allclose(d["loss"], 3.0 * c["loss"], rtol=1e-12)


# --------------------------------------------------------------------------- vocabulary shards
@pytest.mark.parametrize("reduction", REDS)
@pytest.mark.parametrize("cap", [0.0, 2.0])
def test_shard_merge_equals_whole_vocabulary(reduction, cap):
    """Splitting the vocabulary anywhere and merging the shards' (m, d, s, z_y) gives the
    whole-vocabulary results; each shard's backward sums to the whole backward."""
    N, H, V = 23, 9, 61
    hidden, weight, labels = _rand_case(N, H, V, 80, w_std=1.2, ignore=(3, 11))
    whole = orc.forward(hidden, weight, labels, reduction, zloss_coef=0.02, softcap=cap)
    gl, ge = _grads(reduction, N, 80)
    dh_w, dw_w = orc.backward(hidden, weight, labels, whole["lse"], whole["ez"], gl, ge,
                              reduction, zloss_coef=0.02, softcap=cap)
    for cuts in ([0, V], [0, 1, V], [0, 20, 21, 44, V], list(range(0, V + 1, 7)) + [V]):
        cuts = sorted(set(cuts))
        st = np.stack([orc.shard_stats(hidden, weight[:, a:b], labels, a, softcap=cap)
                       for a, b in zip(cuts[:-1], cuts[1:])])
        comb = orc.combine_shards(st, labels, reduction, zloss_coef=0.02, v_total=V)
        np.testing.assert_allclose(comb["lse"], whole["lse"], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(comb["ez"], whole["ez"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(comb["loss"], whole["loss"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(comb["entropy"], whole["entropy"], rtol=1e-12, atol=1e-12)
        dh = np.zeros_like(dh_w)
        for a, b in zip(cuts[:-1], cuts[1:]):
            dhp, dwp = orc.backward(hidden, weight[:, a:b], labels, comb["lse"], comb["ez"], gl,
                                    ge, reduction, zloss_coef=0.02, softcap=cap, v_offset=a,
                                    v_total=V)
            dh += dhp
            np.testing.assert_allclose(dwp, dw_w[:, a:b], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dh, dh_w, rtol=1e-11, atol=1e-13)


def test_extreme_logits_stay_finite():
    """Logits of +-1000 (far past exp's range) give the limits in closed form: the softmax
    puts all mass on the largest logit, lse equals it, the entropy is 0 and the CE of a
    label at -1000 is 2000; the gradients stay finite."""
    hidden = np.array([[1.0]])
    weight = np.array([[1000.0, 0.0, -1000.0]])
    for y, ce in ((0, 0.0), (1, 1000.0), (2, 2000.0)):
        out = orc.forward(hidden, weight, np.array([y]), "none")
        assert out["lse"][0] == 1000.0
        assert out["entropy_tok"][0] == 0.0
        assert out["ce_tok"][0] == ce
        dh, dw = orc.backward(hidden, weight, np.array([y]), out["lse"], out["ez"], [1.0], [1.0],
                              "none")
        assert np.all(np.isfinite(dh)) and np.all(np.isfinite(dw))
        onehot = np.eye(3)[y]
        np.testing.assert_allclose(dw[0], np.eye(3)[0] - onehot, atol=1e-300)


def _random_option_case(i):
    import random
    r = random.Random(600 + i)
    N, H, V = r.randint(1, 6), r.randint(1, 5), r.randint(1, 9)
    hidden, weight, labels = _rand_case(N, H, V, 900 + i, w_std=r.choice([0.3, 0.9, 2.0]),
                                        ignore=tuple(r.sample(range(N), r.randint(0, N))))
    reduction = r.choice(REDS)
    kw = dict(zloss_coef=r.choice([0.0, 0.05]), softcap=r.choice([0.0, 1.5, 4.0]),
              label_smoothing=r.choice([0.0, 0.0, 0.2]))
    cw = np.random.default_rng(950 + i).uniform(0.3, 1.7, V) if r.random() < 0.4 else None
    return hidden, weight, labels, reduction, kw, cw


@pytest.mark.parametrize("i", range(16))
def test_random_options_oracle_against_scalar_loops(i):
    """Seeded random tiny cases over every option at once (reduction, z-loss, soft-cap,
    smoothing, class weights, any set of ignored rows, V down to 1): the oracle's forward
    against the scalar loops, and its backward against central finite differences of
    the scalar-loop objective (a second implementation, not the oracle's own)."""
    hidden, weight, labels, reduction, kw, cw = _random_option_case(i)
    N = hidden.shape[0]
    out = orc.forward(hidden, weight, labels, reduction, class_weight=cw, **kw)
    lkw = dict(kw, class_weight=None if cw is None else cw.tolist())
    l, e, lse = lc.forward_loops(hidden.tolist(), weight.tolist(), labels.tolist(), reduction,
                                 **lkw)
    np.testing.assert_allclose(out["loss"], l, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["entropy"], e, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["lse"], lse, rtol=1e-12)
    gl, ge = _grads(reduction, N, 600 + i)
    dh, dw = orc.backward(hidden, weight, labels, out["lse"], out["ez"], gl, ge, reduction,
                          class_weight=cw, **kw)
    fh, fw = lc.fd_grads_loops(hidden.tolist(), weight.tolist(), labels.tolist(), gl.tolist(),
                               ge.tolist(), reduction=reduction, **lkw)
    np.testing.assert_allclose(dh, np.array(fh), rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(dw, np.array(fw), rtol=1e-5, atol=1e-7)
