"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by
element, on seeded inputs that span several tiles and ragged tails.

Tolerances (the stated bar): per-token loss / entropy / lse / E_p[z] abs err <= 2e-3,
reduced loss and entropy rel err <= 1e-4, dhidden / dweight rel-L2 err <= 1e-2, and
rows with ignore_index contribute exactly 0 (bitwise-zero dhidden rows and per-token
outputs).
"""
import dataclasses

import numpy as np
import pytest
import torch

from linear_cross_entropy_forward_gb300 import flce_backward, flce_forward, linear_cross_entropy
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


def oracle_run(w, hidden, weight, labels, g_loss, g_ent, eps=0.0, cw=None):
    h = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    y = labels.numpy()
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, label_smoothing=eps,
              class_weight=None if cw is None else cw.numpy())
    o = orc.forward(h, W, y, w.reduction, **kw)
    dh, dw = orc.backward(h, W, y, o["lse"], o["ez"], g_loss.numpy(), g_ent.numpy(), w.reduction,
                          **kw)
    return o, dh, dw


def gpu_run(w, hidden, weight, labels, g_loss, g_ent, chunk_v=0, weight_layout="hv", eps=0.0,
            cw=None):
    """weight is [H,V]; with weight_layout 'vh' the GPU gets its [V,H] transpose and the
    returned dw is transposed back to [H,V]."""
    dev = torch.device("cuda")
    hd, yd = hidden.to(dev), labels.to(dev)
    Wd = weight.to(dev) if weight_layout == "hv" else weight.t().contiguous().to(dev)
    kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, weight_layout=weight_layout,
              label_smoothing=eps, class_weight=None if cw is None else cw.to(dev))
    loss, ent, lse, ez = flce_forward(hd, Wd, yd, w.reduction, validate=True, **kw)
    dh, dw = flce_backward(hd, Wd, yd, lse, ez, g_loss.to(dev), g_ent.to(dev), w.reduction,
                           validate=True, chunk_v=chunk_v, **kw)
    torch.cuda.synchronize()
    if weight_layout == "vh":
        assert dw.shape == (w.V, w.H)
        dw = dw.t()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    return dict(loss=f(loss), entropy=f(ent), lse=f(lse), ez=f(ez), dh=f(dh), dw=f(dw),
                dh_raw=dh.cpu())


def check_parity(w, chunk_v=0, report=None, weight_layout="hv", eps=0.0, cw=None):
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    o, dh_o, dw_o = oracle_run(w, hidden, weight, labels, g_loss, g_ent, eps, cw)
    g = gpu_run(w, hidden, weight, labels, g_loss, g_ent, chunk_v, weight_layout, eps, cw)
    valid = o["valid"]
    errs = {}
    errs["lse_abs"] = float(np.abs(g["lse"] - o["lse"]).max())
    errs["ez_abs"] = float(np.abs(g["ez"] - o["ez"]).max())
    if w.reduction == "none":
        errs["loss_tok_abs"] = float(np.abs(g["loss"] - o["loss"]).max())
        errs["ent_tok_abs"] = float(np.abs(g["entropy"] - o["entropy"]).max())
        assert errs["loss_tok_abs"] <= TOK_ABS, errs
        assert errs["ent_tok_abs"] <= TOK_ABS, errs
        assert np.all(g["loss"][~valid] == 0.0) and np.all(g["entropy"][~valid] == 0.0)
    else:
        for k in ("loss", "entropy"):
            ref = float(o[k])
            got = float(g[k][0])
            errs[k + "_rel"] = abs(got - ref) / abs(ref) if ref != 0 else abs(got)
            assert errs[k + "_rel"] <= RED_REL, errs
    assert errs["lse_abs"] <= TOK_ABS, errs
    assert errs["ez_abs"] <= TOK_ABS, errs
    errs["dh_rel_l2"] = rel_l2(g["dh"], dh_o)
    errs["dw_rel_l2"] = rel_l2(g["dw"], dw_o)
    assert errs["dh_rel_l2"] <= GRAD_REL_L2, errs
    assert errs["dw_rel_l2"] <= GRAD_REL_L2, errs
    ign = np.nonzero(~valid)[0]
    if ign.size:
        assert torch.all(g["dh_raw"][torch.from_numpy(ign)].view(torch.int16) == 0)
    if report is not None:
        report.update(errs)
    return errs


W0 = wl.TINY
CASES = [
    # the small workload as specified (mean, 10 % ignored)
    ("tiny", W0, 0),
    # ragged in every dimension: N, H, V not multiples of 128/64/256; several chunks
    ("ragged_none", dataclasses.replace(W0, name="r1", N=300, H=200, V=1000, reduction="none",
                                        grad_mode="normal"), 256),
    ("ragged_mean_zloss", dataclasses.replace(W0, name="r2", N=300, H=200, V=1000,
                                              zloss_coef=1e-3), 512),
    ("sum_zloss", dataclasses.replace(W0, name="r3", N=260, H=128, V=776, reduction="sum",
                                      zloss_coef=1e-2, ignore_frac=0.2), 256),
    # soft-cap that bites (|z'| well above c) and the Gemma-2 value
    ("softcap_tight", dataclasses.replace(W0, name="s1", N=384, H=256, V=2048, w_std=0.3,
                                          softcap=2.0, reduction="none", grad_mode="normal"),
     512),
    ("softcap_30", dataclasses.replace(W0, name="s2", N=256, H=2304 // 4, V=3000 - 8,
                                       w_std=0.03, softcap=30.0), 1024),
    # self-sampled (peaked) labels, RL-style gradients
    ("rl_self_labels", dataclasses.replace(W0, name="q1", N=512, H=448, V=2048, reduction="none",
                                           label_mode="self", grad_mode="rl",
                                           ignore_frac=0.15), 0),
    # one tile, one row, nothing ignored, everything ignored
    ("single_tile", dataclasses.replace(W0, name="t1", N=128, H=64, V=256, reduction="none",
                                        ignore_frac=0.0, grad_mode="normal"), 0),
    ("one_row", dataclasses.replace(W0, name="t2", N=1, H=8, V=8, ignore_frac=0.0), 0),
    ("big_logits", dataclasses.replace(W0, name="t3", N=200, H=512, V=1024, w_std=0.5,
                                       reduction="none", grad_mode="normal"), 0),
    # vocabularies wider than 65536 columns at small N: one backward chunk of 70000
    # columns, and two chunks of 70144 columns (fp32 accumulation of dhidden across them)
    ("dhidden_split", dataclasses.replace(W0, name="d7", N=300, H=64, V=70000,
                                          reduction="none", grad_mode="normal"), 0),
    ("dhidden_split_chunks", dataclasses.replace(W0, name="d8", N=130, H=72, V=140000,
                                                 zloss_coef=1e-3), 70144),
    # a vocabulary of two million columns and a ragged last tile: 8194 tiles per row of
    # forward partials to merge, column indices past 2^21 in every kernel
    ("vocab_2m", dataclasses.replace(W0, name="v2m", N=130, H=64, V=2 ** 21 + 264,
                                     zloss_coef=1e-3), 0),
    # the other extremes: a 16384-wide hidden (256 k-blocks per output tile) and 100000
    # rows (391 row tiles) over a narrow vocabulary
    ("hidden_16k", dataclasses.replace(W0, name="x1", N=300, H=16384, V=1000, w_std=0.004,
                                       reduction="none", grad_mode="normal"), 0),
    ("rows_100k", dataclasses.replace(W0, name="x2", N=100000, H=64, V=264, w_std=0.1,
                                      zloss_coef=1e-3), 256),
]


@pytest.mark.parametrize("name,w,chunk_v", CASES, ids=[c[0] for c in CASES])
def test_parity_small(name, w, chunk_v):
    _cuda_or_skip()
    rep = {}
    check_parity(w, chunk_v, rep)
    print(name, rep)


VH_CASES = [c for c in CASES if c[0] in ("tiny", "ragged_none", "ragged_mean_zloss",
                                          "softcap_tight", "single_tile", "one_row")]


@pytest.mark.parametrize("name,w,chunk_v", VH_CASES, ids=[c[0] for c in VH_CASES])
def test_parity_weight_vh(name, w, chunk_v):
    """Weight stored [V,H] (nn.Linear layout): same results as the [H,V] oracle."""
    _cuda_or_skip()
    rep = {}
    check_parity(w, chunk_v, rep, weight_layout="vh")
    print(name, "vh", rep)


# A [V,H] weight takes any vocabulary size: V is not a row length there, so it needs no
# multiple of 8 (the [H,V] layout does).  GPT-2's 50257 among them.
VH_ODD_VOCAB_CASES = [
    ("odd_none_chunks", dataclasses.replace(W0, name="o1", N=300, H=200, V=1001,
                                            reduction="none", grad_mode="normal"), 256),
    ("gpt2_vocab_mean_zloss", dataclasses.replace(W0, name="o2", N=256, H=256, V=50257,
                                                  zloss_coef=1e-4), 0),
    ("odd_softcap_sum", dataclasses.replace(W0, name="o3", N=130, H=64, V=777, w_std=0.3,
                                            softcap=3.0, reduction="sum"), 256),
    ("one_class_column_past_tile", dataclasses.replace(W0, name="o4", N=64, H=16, V=257,
                                                       ignore_frac=0.0), 0),
    # the degenerate vocabularies: one class (CE = entropy = 0; only the z-loss has a
    # gradient) and two
    ("single_class_zloss", dataclasses.replace(W0, name="o6", N=37, H=16, V=1,
                                               zloss_coef=1e-2), 0),
    ("two_classes_none", dataclasses.replace(W0, name="o7", N=300, H=24, V=2, w_std=0.5,
                                             reduction="none", grad_mode="normal"), 0),
]


@pytest.mark.parametrize("name,w,chunk_v", VH_ODD_VOCAB_CASES,
                         ids=[c[0] for c in VH_ODD_VOCAB_CASES])
def test_parity_weight_vh_any_vocabulary_size(name, w, chunk_v):
    _cuda_or_skip()
    rep = {}
    check_parity(w, chunk_v, rep, weight_layout="vh")
    print(name, "vh", rep)


def test_parity_weight_vh_odd_vocabulary_smoothing_and_class_weights():
    _cuda_or_skip()
    w = dataclasses.replace(W0, name="o5", N=300, H=200, V=999, reduction="mean")
    cw = torch.rand(w.V, generator=torch.Generator().manual_seed(5)) * 1.5 + 0.25
    check_parity(w, 256, {}, weight_layout="vh", eps=0.1, cw=cw)


def test_hv_weight_refuses_a_vocabulary_that_is_not_a_multiple_of_8():
    _cuda_or_skip()
    from linear_cross_entropy_forward_gb300 import FlceError
    dev = torch.device("cuda")
    h = torch.zeros(4, 16, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(4, dtype=torch.int64, device=dev)
    with pytest.raises(FlceError) as ei:
        flce_forward(h, torch.zeros(16, 1001, dtype=torch.bfloat16, device=dev), y, "mean")
    assert ei.value.code == 3


SMOOTH_CASES = [
    # (name, workload, chunk_v, label_smoothing, class weights?)
    ("smooth_mean", dataclasses.replace(W0, name="ls1", N=300, H=200, V=1000), 256, 0.1, False),
    ("weights_mean", dataclasses.replace(W0, name="ls2", N=300, H=200, V=1000), 512, 0.0, True),
    ("smooth_weights_none", dataclasses.replace(W0, name="ls3", N=260, H=128, V=776,
                                                reduction="none", grad_mode="normal"),
     256, 0.2, True),
    ("smooth_weights_sum_zloss_cap", dataclasses.replace(W0, name="ls4", N=384, H=256, V=2048,
                                                         reduction="sum", zloss_coef=1e-2,
                                                         softcap=3.0, w_std=0.2), 512, 0.05, True),
    ("smooth_weights_mean_zloss", dataclasses.replace(W0, name="ls5", N=256, H=512, V=4096,
                                                      zloss_coef=1e-4), 0, 0.1, True),
]


@pytest.mark.parametrize("name,w,chunk_v,eps,weighted", SMOOTH_CASES,
                         ids=[c[0] for c in SMOOTH_CASES])
def test_parity_smoothing_and_class_weights(name, w, chunk_v, eps, weighted):
    _cuda_or_skip()
    cw = None
    if weighted:
        g = torch.Generator().manual_seed(123)
        cw = torch.rand(w.V, generator=g) * 1.5 + 0.25
    rep = {}
    check_parity(w, chunk_v, rep, eps=eps, cw=cw)
    print(name, rep)


def test_layouts_agree_bitwise():
    """The two weight layouts run kernels with different operand-major descriptors,
    but the UMMAs sum the same products in the same K order: identical results."""
    _cuda_or_skip()
    w = dataclasses.replace(W0, name="lay", N=300, H=200, V=1000, zloss_coef=1e-3,
                            softcap=5.0)
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    a = gpu_run(w, hidden, weight, labels, g_loss, g_ent, 256, "hv")
    b = gpu_run(w, hidden, weight, labels, g_loss, g_ent, 256, "vh")
    for k in ("loss", "entropy", "lse", "ez", "dh", "dw"):
        assert np.array_equal(a[k], b[k]), k


def test_all_ignored_mean_is_zero():
    _cuda_or_skip()
    w = dataclasses.replace(W0, name="t4", N=200, H=64, V=512, ignore_frac=1.0)
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    g = gpu_run(w, hidden, weight, labels, g_loss, g_ent)
    assert g["loss"][0] == 0.0 and g["entropy"][0] == 0.0
    assert not np.any(g["dh"]) and not np.any(g["dw"])


def test_zero_rows():
    _cuda_or_skip()
    dev = torch.device("cuda")
    hidden = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    weight = torch.randn(64, 256, device=dev).to(torch.bfloat16)
    labels = torch.empty(0, dtype=torch.int64, device=dev)
    loss, ent, lse, ez = flce_forward(hidden, weight, labels, "mean", validate=True)
    assert loss.item() == 0.0 and ent.item() == 0.0
    dh, dw = flce_backward(hidden, weight, labels, lse, ez, torch.ones(1, device=dev),
                           torch.ones(1, device=dev), "mean", validate=True)
    assert dh.shape == (0, 64) and not torch.any(dw)


def test_bad_label_reported():
    _cuda_or_skip()
    from linear_cross_entropy_forward_gb300 import FlceError
    dev = torch.device("cuda")
    hidden = torch.randn(64, 64, device=dev).to(torch.bfloat16)
    weight = torch.randn(64, 256, device=dev).to(torch.bfloat16)
    labels = torch.zeros(64, dtype=torch.int64, device=dev)
    labels[5] = 256  # out of range and not ignore_index
    with pytest.raises(FlceError) as ei:
        flce_forward(hidden, weight, labels, "none", validate=True)
    assert ei.value.code == 5


def test_bad_labels_flag_only_their_rows():
    """Labels outside [0, V) that are not ignore_index (past V, far past it, negative):
    without validate the call still completes, the workspace's status reports
    FLCE_ERR_LABEL, those rows' loss and entropy are NaN, and every other output (the
    other rows' loss and entropy, every row's lse and E_p[z]) matches the oracle."""
    _cuda_or_skip()
    from linear_cross_entropy_forward_gb300 import flce_status, make_params, workspace_size
    w = dataclasses.replace(W0, name="bl", N=300, H=64, V=1000, reduction="none",
                            grad_mode="normal")
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    bad_rows = [3, 77, 150, 151, 299]
    bad = labels.clone()
    for r_, v in zip(bad_rows, [w.V, w.V + 7, -5, -101, 1 << 40]):
        bad[r_] = v
    dev = torch.device("cuda")
    ws = torch.empty(workspace_size(make_params(w.N, w.H, w.V, "none"), 0), dtype=torch.uint8,
                     device=dev)
    loss, ent, lse, ez = flce_forward(hidden.to(dev), weight.to(dev), bad.to(dev), "none",
                                      workspace=ws)
    assert flce_status(ws) == 5
    h = orc.bf16_bits_to_f64(wl.bf16_bits(hidden))
    W = orc.bf16_bits_to_f64(wl.bf16_bits(weight))
    masked = bad.numpy().copy()
    masked[bad_rows] = orc.IGNORE_INDEX
    o = orc.forward(h, W, masked, "none")
    f = lambda t: t.cpu().numpy().astype(np.float64)  # noqa: E731
    good = np.ones(w.N, bool)
    good[bad_rows] = False
    assert np.all(np.isnan(f(loss)[bad_rows])) and np.all(np.isnan(f(ent)[bad_rows]))
    assert np.abs(f(loss)[good] - o["loss"][good]).max() <= TOK_ABS
    assert np.abs(f(ent)[good] - o["entropy"][good]).max() <= TOK_ABS
    assert np.abs(f(lse) - o["lse"]).max() <= TOK_ABS
    assert np.abs(f(ez) - o["ez"]).max() <= TOK_ABS


def test_deterministic_repeat():
    _cuda_or_skip()
    w = dataclasses.replace(W0, name="d1", N=300, H=200, V=1000, zloss_coef=1e-3)
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    a = gpu_run(w, hidden, weight, labels, g_loss, g_ent, 256)
    b = gpu_run(w, hidden, weight, labels, g_loss, g_ent, 256)
    for k in ("loss", "entropy", "lse", "ez", "dh", "dw"):
        assert np.array_equal(a[k], b[k]), k


def test_autograd_function_matches_explicit_calls():
    _cuda_or_skip()
    dev = torch.device("cuda")
    w = dataclasses.replace(W0, name="a1", N=256, H=128, V=1024)
    hidden, weight, labels, _, _ = wl.make_inputs(w)
    h = hidden.to(dev).requires_grad_(True)
    W = weight.to(dev).requires_grad_(True)
    y = labels.to(dev)
    loss, ent = linear_cross_entropy(h, W, y, reduction="mean")
    (loss + 0.5 * ent).backward()
    _, _, lse, ez = flce_forward(h.detach(), W.detach(), y, "mean")
    dh, dw = flce_backward(h.detach(), W.detach(), y, lse, ez, torch.ones(1, device=dev),
                           torch.full((1,), 0.5, device=dev), "mean")
    assert torch.equal(h.grad, dh) and torch.equal(W.grad, dw)


def test_binding_rejects_mismatched_outputs_and_workspace():
    """Caller-provided outputs and workspaces are checked on the host before any launch."""
    _cuda_or_skip()
    from linear_cross_entropy_forward_gb300 import flce_forward_backward
    dev = torch.device("cuda")
    hidden = torch.randn(64, 64, device=dev).to(torch.bfloat16)
    weight = torch.randn(64, 256, device=dev).to(torch.bfloat16)
    labels = torch.zeros(64, dtype=torch.int64, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    good = (torch.empty(64, **f32), torch.empty(64, **f32), torch.empty(64, **f32),
            torch.empty(64, **f32))
    flce_forward(hidden, weight, labels, "none", out=good)
    with pytest.raises(ValueError):  # wrong shape
        flce_forward(hidden, weight, labels, "none", out=(good[0][:32],) + good[1:])
    with pytest.raises(TypeError):  # wrong dtype
        flce_forward(hidden, weight, labels, "none",
                     out=(good[0].double(),) + good[1:])
    with pytest.raises(ValueError):  # too few tensors
        flce_forward(hidden, weight, labels, "none", out=good[:3])
    with pytest.raises(TypeError):  # workspace not bytes
        flce_forward(hidden, weight, labels, "none", workspace=torch.empty(1 << 20, **f32))
    with pytest.raises(ValueError):  # a workspace too small is refused, not replaced
        flce_forward(hidden, weight, labels, "none",
                     workspace=torch.empty(256, dtype=torch.uint8, device=dev))
    dh = torch.empty(64, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):  # dweight shaped like dhidden
        flce_backward(hidden, weight, labels, good[2], good[3], None, None, "none",
                      out=(dh, torch.empty(64, 64, dtype=torch.bfloat16, device=dev)))
    with pytest.raises(ValueError):
        flce_forward_backward(hidden, weight, labels, None, None, "mean",
                              out=(torch.empty(64, **f32),) * 4 + (dh, dh))
    with pytest.raises(TypeError):  # a CPU tensor among CUDA ones
        flce_forward(hidden, weight, labels.cpu(), "none")


def test_schedule_counters_are_zero_after_every_call():
    """The GEMMs draw their tiles from pairs of counters in the workspace header (bytes
    128-135 for the caller's stream, 136-143 for dweight running beside dhidden); the last
    CTA pair of each GEMM resets its pair, so after a call that ran many GEMMs on one
    workspace (a backward of four vocabulary chunks: 12 GEMMs; a gradient-in-forward call
    of three token chunks: 9) they are zero again, and results are right."""
    _cuda_or_skip()
    from linear_cross_entropy_forward_gb300 import (flce_forward_backward, make_params,
                                                    workspace_size)
    dev = torch.device("cuda")
    w = dataclasses.replace(W0, name="sc", N=1100, H=200, V=1000, reduction="none",
                            grad_mode="normal")
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(w)
    hd, Wd, yd = hidden.to(dev), weight.to(dev), labels.to(dev)
    gl, ge = g_loss.to(dev), g_ent.to(dev)
    p1 = make_params(w.N, w.H, w.V, "none", chunk_v=256)
    ws_f = torch.full((workspace_size(p1, 0),), 7, dtype=torch.uint8, device=dev)
    ws_b = torch.full((workspace_size(p1, 1),), 7, dtype=torch.uint8, device=dev)
    p3 = make_params(w.N, w.H, w.V, "none", chunk_n=512)
    ws_g = torch.full((workspace_size(p3, 3),), 7, dtype=torch.uint8, device=dev)
    for _ in range(2):  # the second round starts from the counters the first left
        _, _, lse, ez = flce_forward(hd, Wd, yd, "none", validate=True, workspace=ws_f)
        dh, dw = flce_backward(hd, Wd, yd, lse, ez, gl, ge, "none", validate=True, chunk_v=256,
                               workspace=ws_b)
        out = flce_forward_backward(hd, Wd, yd, gl, ge, "none", validate=True, chunk_n=512,
                                    workspace=ws_g)
        torch.cuda.synchronize()
        for ws in (ws_f, ws_b, ws_g):
            assert torch.all(ws[128:144] == 0), ws[128:144].tolist()
    o, dh_o, dw_o = oracle_run(w, hidden, weight, labels, g_loss, g_ent)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    assert rel_l2(f(dh), dh_o) <= GRAD_REL_L2 and rel_l2(f(dw), dw_o) <= GRAD_REL_L2
    assert rel_l2(f(out[4]), dh_o) <= GRAD_REL_L2 and rel_l2(f(out[5]), dw_o) <= GRAD_REL_L2


def test_one_dirty_workspace_shared_by_many_problems():
    """The workspace is scratch: one buffer, filled with a different garbage byte before
    every use, shared by a sequence of different problems (both layouts, several
    chunkings, both modes), gives every call the bits a fresh workspace gives."""
    import random
    from linear_cross_entropy_forward_gb300 import flce_forward_backward
    _cuda_or_skip()
    dev = torch.device("cuda")
    big = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for i in range(12):
        r = random.Random(97000 + i)
        layout = r.choice(["hv", "vh"])
        V = r.randint(1, 3000) if layout == "vh" else 8 * r.randint(1, 375)
        gif = r.random() < 0.4
        red = r.choice(["mean", "sum", "none"])
        w = dataclasses.replace(W0, name=f"ws{i}", seed=970 + i, N=r.choice([1, 37, 300, 1100]),
                                H=8 * r.randint(1, 64), V=V, reduction=red,
                                zloss_coef=r.choice([0.0, 1e-3]), softcap=r.choice([0.0, 5.0]),
                                grad_mode="normal" if red == "none" else "ones")
        h, W, y, gl, ge = wl.make_inputs(w)
        if layout == "vh":
            W = W.t().contiguous()
        hd, Wd, yd, gld, ged = (x.to(dev) for x in (h, W, y, gl, ge))
        kw = dict(zloss_coef=w.zloss_coef, softcap=w.softcap, weight_layout=layout)
        chunk_v = r.choice([0, 256])
        results = []
        for ws in (None, big):
            big.fill_(r.randint(0, 255))
            if gif:
                results.append(flce_forward_backward(hd, Wd, yd, gld, ged, red, workspace=ws,
                                                     **kw))
            else:
                f = flce_forward(hd, Wd, yd, red, workspace=ws, **kw)
                results.append((*f, *flce_backward(hd, Wd, yd, f[2], f[3], gld, ged, red,
                                                   chunk_v=chunk_v, workspace=ws, **kw)))
            torch.cuda.synchronize()
        for a, b in zip(*results):
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), (i, w, layout, gif, chunk_v)
