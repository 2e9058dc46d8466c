"""Scalar-loop brute-force checker (pure Python, math module).  TEST INFRASTRUCTURE ONLY.

An independent second implementation of the forward values, written with plain
loops so a reader can check each line against the definitions of verl PR #462
("Equivalent compute logic"), Liger-Kernel PR #435 (reduction, z-loss) and
Liger-Kernel issue #127 (soft-cap).  It is meant for tiny inputs (a few rows,
tens of columns) and pins the vectorised oracle.  Gradients here come from
central finite differences of these loops, not from any closed form.
"""
from __future__ import annotations

import math

IGNORE_INDEX = -100


def forward_loops(hidden, weight, labels, reduction="mean", ignore_index=IGNORE_INDEX,
                  zloss_coef=0.0, softcap=0.0, label_smoothing=0.0, class_weight=None):
    """hidden: list of N lists of H floats; weight: H lists of V floats; labels: N ints.

    With label smoothing eps and class weights w (torch's cross_entropy definition):
    the cross-entropy of a token is (1 - eps) w_y (-log p_y) + eps/V sum_c w_c (-log p_c),
    and the mean divides it by the summed w_y of the non-ignored tokens."""
    N = len(hidden)
    H = len(weight)
    V = len(weight[0])
    w = class_weight if class_weight is not None else [1.0] * V
    eps = label_smoothing
    ce_tok, zl_tok, loss_tok, ent_tok, lse_all = [], [], [], [], []
    n_valid = 0
    w_valid = 0.0
    for n in range(N):
        z = []
        for v in range(V):
            acc = 0.0
            for h in range(H):
                acc += hidden[n][h] * weight[h][v]
            if softcap != 0.0:
                acc = softcap * math.tanh(acc / softcap)
            z.append(acc)
        mx = max(z)
        tot = sum(math.exp(zi - mx) for zi in z)
        lse = mx + math.log(tot)
        p = [math.exp(zi - lse) for zi in z]
        # Shannon entropy of the softmax, -sum p log p
        ent = -sum(pi * math.log(pi) for pi in p if pi > 0.0)
        lse_all.append(lse)
        y = labels[n]
        if y == ignore_index:
            ce_tok.append(0.0)
            zl_tok.append(0.0)
            loss_tok.append(0.0)
            ent_tok.append(0.0)
            continue
        n_valid += 1
        w_valid += w[y]
        smooth = 0.0
        for c in range(V):
            smooth += w[c] * -math.log(p[c])
        ce = (1.0 - eps) * w[y] * -math.log(p[y]) + eps / V * smooth
        zl = zloss_coef * lse * lse
        ce_tok.append(ce)
        zl_tok.append(zl)
        loss_tok.append(ce + zl)
        ent_tok.append(ent)
    if reduction == "none":
        return loss_tok, ent_tok, lse_all
    if reduction == "sum":
        return sum(loss_tok), sum(ent_tok), lse_all
    loss = (sum(ce_tok) / w_valid if w_valid != 0 else 0.0) + \
        (sum(zl_tok) / n_valid if n_valid else 0.0)
    ent_mean = sum(ent_tok) / n_valid if n_valid else 0.0
    return loss, ent_mean, lse_all


def objective_loops(hidden, weight, labels, g_loss, g_entropy, reduction="mean",
                    ignore_index=IGNORE_INDEX, zloss_coef=0.0, softcap=0.0,
                    label_smoothing=0.0, class_weight=None):
    l, e, _ = forward_loops(hidden, weight, labels, reduction, ignore_index, zloss_coef, softcap,
                            label_smoothing, class_weight)
    if reduction == "none":
        return sum(g * x for g, x in zip(g_loss, l)) + sum(g * x for g, x in zip(g_entropy, e))
    return g_loss[0] * l + g_entropy[0] * e


def fd_grads_loops(hidden, weight, labels, g_loss, g_entropy, eps=1e-5, **kw):
    """Central finite differences of objective_loops w.r.t. every hidden and weight entry."""
    import copy
    N, H, V = len(hidden), len(weight), len(weight[0])
    dh = [[0.0] * H for _ in range(N)]
    dw = [[0.0] * V for _ in range(H)]
    for n in range(N):
        for h in range(H):
            hp = copy.deepcopy(hidden)
            hm = copy.deepcopy(hidden)
            hp[n][h] += eps
            hm[n][h] -= eps
            dh[n][h] = (objective_loops(hp, weight, labels, g_loss, g_entropy, **kw)
                        - objective_loops(hm, weight, labels, g_loss, g_entropy, **kw)) / (2 * eps)
    for h in range(H):
        for v in range(V):
            wp = copy.deepcopy(weight)
            wm = copy.deepcopy(weight)
            wp[h][v] += eps
            wm[h][v] -= eps
            dw[h][v] = (objective_loops(hidden, wp, labels, g_loss, g_entropy, **kw)
                        - objective_loops(hidden, wm, labels, g_loss, g_entropy, **kw)) / (2 * eps)
    return dh, dw
