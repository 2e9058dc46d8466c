"""fp64 CPU oracle for fused linear cross-entropy + entropy.  TEST INFRASTRUCTURE ONLY.

Nothing on the product path may import this module: only the tests, the smoke
check and the benchmark's CPU-baseline leg use it.  It shares no code with the
CUDA library.

What it computes (plain definitions, written out in fp64):

* verl PR #462, "Equivalent compute logic": logits = hidden @ weight in wide
  precision, p = softmax(logits), entropy = logsumexp(logits) - sum(p * logits),
  and the cross-entropy of the labelled token (the page returns its negation,
  a log-probability).
* Liger-Kernel PR #551 (review by qingquansong): ignored tokens are left out and
  the mean divides by the number of non-ignored tokens, for the entropy term too.
* Liger-Kernel PR #435, "Summary" / "Changes Made": reduction 'none' returns the
  per-token vector; the z-loss follows the same reduction.  The z-loss formula
  is not printed; this oracle takes z_n = coef * lse_n^2 added to the loss.
* Liger-Kernel issue #127 (troy1729, qingquansong): the Gemma-2 soft-cap is
  applied to the logits after the matmul in three steps (divide by c, tanh,
  multiply by c); its backward follows from the chain rule, d tanh(x)/dx =
  1 - tanh(x)^2.
* Liger-Kernel PR #551 (review): label smoothing and per-class target weights
  are further options of the same loss.  Their definition here is torch's
  cross_entropy(weight=w, label_smoothing=eps): the cross-entropy part of a
  token is (1 - eps) w_y (lse - z_y) + (eps / V) sum_c w_c (lse - z_c), and the
  mean divides it by the sum of w_y over non-ignored tokens.  The z-loss and the
  entropy stay unweighted and their mean divides by the non-ignored count
  (the review asks for n_non_ignore in the entropy term).

Backward (closed form of the derivative of the objective
J = sum_n gl_n * loss_n + ge_n * entropy_n, with gl/ge the upstream gradients
after the reduction's scaling and zero on ignored rows; without smoothing and
weights):
    dz_nv = gl_n * (p_nv - [v == y_n] + 2 coef lse_n p_nv) - ge_n * p_nv * (z_nv - E_p[z]_n)
With smoothing eps and class weights w (W = sum_c w_c), the cross-entropy part
contributes a_n (p_nv ((1 - eps) w_y + eps W / V) - (1 - eps) w_y [v == y_n] - eps w_v / V).
    dz'_nv = dz_nv * (1 - (z_nv / c)^2)            (soft-cap on)
    dhidden = dz' @ weight^T,   dweight = hidden^T @ dz'

Every function works over vocabulary chunks so no [N, V] array is formed for
the large shapes.  The maximum and the sums are taken in two passes (not an
online recurrence), so the oracle follows the definitions as written.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100
_REDS = ("none", "mean", "sum")


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) to float64, exactly.

    A bf16 value is the upper half of an IEEE binary32, so shifting the bits
    left by 16 gives the binary32 value, which float64 holds exactly.
    """
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _cap(zp: np.ndarray, softcap: float) -> np.ndarray:
    """Liger-Kernel issue #127: divide by c, tanh, multiply by c (off when c == 0)."""
    if softcap == 0.0:
        return zp
    return softcap * np.tanh(zp / softcap)


def _class_weights(class_weight, V):
    if class_weight is None:
        return np.ones(V)
    w = np.asarray(class_weight, dtype=np.float64).reshape(-1)
    if w.shape != (V,):
        raise ValueError("class_weight must have V entries")
    return w


def _check(hidden, weight, labels, reduction, ignore_index, v_total=None):
    if reduction not in _REDS:
        raise ValueError(f"reduction must be one of {_REDS}")
    N, H = hidden.shape
    H2, V = weight.shape
    if H != H2 or labels.shape != (N,):
        raise ValueError("shape mismatch")
    lab = np.asarray(labels, dtype=np.int64)
    valid = lab != ignore_index
    if np.any((lab[valid] < 0) | (lab[valid] >= (V if v_total is None else v_total))):
        raise ValueError("label out of range")
    return N, H, V, lab, valid


def logits_chunk(hidden: np.ndarray, weight: np.ndarray, v0: int, v1: int,
                 softcap: float = 0.0) -> np.ndarray:
    """Capped logits z[:, v0:v1] = cap(hidden @ weight[:, v0:v1]) in fp64."""
    return _cap(hidden @ weight[:, v0:v1], softcap)


def row_stats(hidden, weight, softcap=0.0, v_chunk=8192, class_weight=None):
    """Per-row log-sum-exp, softmax mean and class-weighted sum of the capped logits.

    Pass 1: m_n = max_v z_nv.  Pass 2: d_n = sum_v exp(z_nv - m_n) and
    s_n = sum_v exp(z_nv - m_n) * z_nv.  Then lse = m + log d, E_p[z] = s / d.
    Also sw_n = sum_v w_v z_nv (w = class_weight, ones by default).
    """
    N = hidden.shape[0]
    V = weight.shape[1]
    m = np.full(N, -np.inf)
    for v0 in range(0, V, v_chunk):
        z = logits_chunk(hidden, weight, v0, min(V, v0 + v_chunk), softcap)
        m = np.maximum(m, z.max(axis=1))
    cw = _class_weights(class_weight, V)
    d = np.zeros(N)
    s = np.zeros(N)
    sw = np.zeros(N)
    for v0 in range(0, V, v_chunk):
        v1 = min(V, v0 + v_chunk)
        z = logits_chunk(hidden, weight, v0, v1, softcap)
        e = np.exp(z - m[:, None])
        d += e.sum(axis=1)
        s += (e * z).sum(axis=1)
        sw += z @ cw[v0:v1]
    lse = m + np.log(d)
    ez = s / d
    return lse, ez, sw


def label_logits(hidden, weight, labels, valid, softcap=0.0):
    """z_{n, y_n} for non-ignored rows (0 elsewhere)."""
    zy = np.zeros(hidden.shape[0])
    idx = np.nonzero(valid)[0]
    if idx.size:
        zp = np.einsum("nh,hn->n", hidden[idx], weight[:, labels[idx]])
        zy[idx] = _cap(zp, softcap)
    return zy


def forward(hidden, weight, labels, reduction="mean", ignore_index=IGNORE_INDEX,
            zloss_coef=0.0, softcap=0.0, v_chunk=8192, label_smoothing=0.0, class_weight=None,
            stats=None):
    """Loss and entropy of verl PR #462's compute logic, with the Liger options.

    ``stats``: the (lse, ez, sw) that :func:`row_stats` returns for these hidden,
    weight, softcap and class_weight, when the caller already has them (they do not
    depend on the labels); None computes them here.

    Returns a dict:
      loss, entropy   -- reduced ('mean'/'sum': float; 'none': [N] arrays)
      loss_tok, entropy_tok -- per-token values, 0 on ignored rows
      ce_tok          -- per-token cross-entropy (0 on ignored rows); logprob = -ce
      lse, ez         -- per-row log-sum-exp and E_p[z] for every row (saved for backward)
      n_valid         -- number of non-ignored rows
    """
    hidden = np.asarray(hidden, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    N, H, V, lab, valid = _check(hidden, weight, labels, reduction, ignore_index)
    cw = _class_weights(class_weight, V)
    eps = float(label_smoothing)
    if stats is None:
        stats = row_stats(hidden, weight, softcap, v_chunk, class_weight)
    lse, ez, sw = (np.asarray(a, dtype=np.float64) for a in stats)
    if lse.shape != (N,) or ez.shape != (N,) or sw.shape != (N,):
        raise ValueError("stats must hold three [N] arrays")
    zy = label_logits(hidden, weight, lab, valid, softcap)
    wy = np.where(valid, cw[np.where(valid, lab, 0)], 0.0)
    # cross-entropy part: (1 - eps) w_y (lse - z_y) + eps/V (W lse - sum_c w_c z_c)
    ce = np.where(valid, (1.0 - eps) * wy * (lse - zy) + (eps / V) * (cw.sum() * lse - sw), 0.0)
    ent = np.where(valid, lse - ez, 0.0)
    zl = np.where(valid, zloss_coef * lse * lse, 0.0)
    loss_tok = ce + zl
    n_valid = int(valid.sum())
    w_valid = float(wy.sum())
    if reduction == "none":
        loss, entropy = loss_tok, ent
    elif reduction == "sum":
        loss, entropy = float(loss_tok.sum()), float(ent.sum())
    else:
        # mean over non-ignored tokens (the cross-entropy part over their summed class
        # weights); an all-ignored batch reduces to 0
        loss = (float(ce.sum()) / w_valid if w_valid != 0 else 0.0) + \
            (float(zl.sum()) / n_valid if n_valid > 0 else 0.0)
        entropy = float(ent.sum()) / n_valid if n_valid > 0 else 0.0
    return dict(loss=loss, entropy=entropy, loss_tok=loss_tok, entropy_tok=ent, ce_tok=ce,
                lse=lse, ez=ez, n_valid=n_valid, valid=valid, w_valid=w_valid)


def grad_scales(g_loss, g_entropy, valid, reduction, w_valid=None):
    """Per-row upstream gradients after the reduction, zero on ignored rows:
    (gl_ce, gl_z, ge) = g (none/sum); for mean the cross-entropy part's is divided
    by the summed class weights w_valid (the non-ignored count without weights),
    the z-loss and entropy parts' by the non-ignored count."""
    N = valid.shape[0]
    gl = np.broadcast_to(np.asarray(g_loss, dtype=np.float64).reshape(-1), (N,)).copy()
    ge = np.broadcast_to(np.asarray(g_entropy, dtype=np.float64).reshape(-1), (N,)).copy()
    gc = gl.copy()
    if reduction == "mean":
        n_valid = int(valid.sum())
        s = 1.0 / n_valid if n_valid > 0 else 0.0
        wv = float(n_valid) if w_valid is None else float(w_valid)
        gc *= 1.0 / wv if wv != 0 else 0.0
        gl *= s
        ge *= s
    gc[~valid] = 0.0
    gl[~valid] = 0.0
    ge[~valid] = 0.0
    return gc, gl, ge


def dlogits_chunk(hidden, weight, labels, lse, ez, gc, gl, ge, v0, v1,
                  zloss_coef=0.0, softcap=0.0, label_smoothing=0.0, class_weight=None,
                  v_offset=0):
    """Gradient of the objective w.r.t. the raw (pre-cap) logits z'[:, v0:v1]
    (gc, gl, ge: per-row scaled upstream grads of the cross-entropy part, the
    z-loss part and the entropy, from grad_scales).  Column v of weight is the
    vocabulary entry v_offset + v (a vocabulary shard)."""
    V = weight.shape[1]
    cw = _class_weights(class_weight, V)
    eps = float(label_smoothing)
    z = logits_chunk(hidden, weight, v0, v1, softcap)
    p = np.exp(z - lse[:, None])
    onehot = (labels[:, None] == np.arange(v_offset + v0, v_offset + v1)[None, :]
              ).astype(np.float64)
    wy = cw[np.clip(labels, 0, V - 1)][:, None]
    ce_grad = p * ((1.0 - eps) * wy + eps * cw.sum() / V) - (1.0 - eps) * wy * onehot \
        - (eps / V) * cw[v0:v1][None, :]
    dz = gc[:, None] * ce_grad + gl[:, None] * 2.0 * zloss_coef * lse[:, None] * p \
        - ge[:, None] * p * (z - ez[:, None])
    if softcap != 0.0:
        dz = dz * (1.0 - (z / softcap) ** 2)
    return dz


def backward(hidden, weight, labels, lse, ez, g_loss, g_entropy, reduction="mean",
             ignore_index=IGNORE_INDEX, zloss_coef=0.0, softcap=0.0, v_chunk=8192,
             rows=None, label_smoothing=0.0, class_weight=None, v_offset=0, v_total=None,
             cols=None):
    """(dhidden, dweight) in fp64.

    ``lse``/``ez`` must come from :func:`forward` on the same inputs.  With
    ``rows`` given, only dhidden[rows] is formed (dweight is then None): each
    dhidden row needs only its own row of the logits.  With ``cols`` given, only
    the columns dweight[:, cols] are formed, over every row (dhidden is then None):
    each dweight column needs only its own column of the logits, and every row's
    lse and E_p[z].  With a vocabulary shard
    (weight = columns [v_offset, v_offset + V) of v_total, lse / ez of the whole
    vocabulary) the result is the shard's dweight and its term of dhidden.
    """
    hidden = np.asarray(hidden, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    N, H, V, lab, valid = _check(hidden, weight, labels, reduction, ignore_index, v_total)
    if v_total is not None and (label_smoothing != 0.0 or class_weight is not None):
        raise ValueError("vocabulary shards exclude label smoothing and class weights")
    cw = _class_weights(class_weight, V)
    w_valid = float(np.where(valid, cw[np.where(valid, lab, 0)], 0.0).sum()) \
        if class_weight is not None else float(valid.sum())
    gc, gl, ge = grad_scales(g_loss, g_entropy, valid, reduction, w_valid)
    opts = dict(zloss_coef=zloss_coef, softcap=softcap, label_smoothing=label_smoothing,
                class_weight=class_weight, v_offset=v_offset)
    if rows is not None and cols is not None:
        raise ValueError("give rows or cols, not both")
    if cols is not None:
        cols = np.asarray(cols, dtype=np.int64).reshape(-1)
        if np.any((cols < 0) | (cols >= V)):
            raise ValueError("column out of range")
        dw = np.zeros((H, cols.size))
        for i, c in enumerate(cols):
            dz = dlogits_chunk(hidden, weight, lab, lse, ez, gc, gl, ge, int(c), int(c) + 1,
                               **opts)
            dw[:, i] = hidden.T @ dz[:, 0]
        return None, dw
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        hs, ls, vs = hidden[rows], lab[rows], valid[rows]
        dh = np.zeros((rows.size, H))
        for v0 in range(0, V, v_chunk):
            v1 = min(V, v0 + v_chunk)
            dz = dlogits_chunk(hs, weight, ls, lse[rows], ez[rows], gc[rows], gl[rows], ge[rows],
                               v0, v1, **opts)
            dh += dz @ weight[:, v0:v1].T
        return dh, None
    dh = np.zeros((N, H))
    dw = np.zeros((H, V))
    for v0 in range(0, V, v_chunk):
        v1 = min(V, v0 + v_chunk)
        dz = dlogits_chunk(hidden, weight, lab, lse, ez, gc, gl, ge, v0, v1, **opts)
        dh += dz @ weight[:, v0:v1].T
        dw[:, v0:v1] = hidden.T @ dz
    return dh, dw


def objective(hidden, weight, labels, g_loss, g_entropy, reduction="mean",
              ignore_index=IGNORE_INDEX, zloss_coef=0.0, softcap=0.0, label_smoothing=0.0,
              class_weight=None):
    """J = <g_loss, loss> + <g_entropy, entropy> (scalar), the function whose gradient
    :func:`backward` returns.  Used for finite-difference pins."""
    out = forward(hidden, weight, labels, reduction, ignore_index, zloss_coef, softcap,
                  label_smoothing=label_smoothing, class_weight=class_weight)
    gl = np.asarray(g_loss, dtype=np.float64).reshape(-1)
    ge = np.asarray(g_entropy, dtype=np.float64).reshape(-1)
    if reduction == "none":
        return float(np.dot(gl * np.ones_like(out["loss"]), out["loss"])
                     + np.dot(ge * np.ones_like(out["entropy"]), out["entropy"]))
    return float(gl[0] * out["loss"] + ge[0] * out["entropy"])


# --------------------------------------------------------------------------- vocabulary shards
def shard_stats(hidden, weight, labels, v_offset, softcap=0.0, v_chunk=8192):
    """Softmax statistics of one vocabulary shard (weight = columns [v_offset, v_offset + V)
    of the whole vocabulary), two passes: m = max z, d = sum exp(z - m),
    s = sum exp(z - m) z, and the label's logit z_y when the label is in the shard
    (0 otherwise).  Returns a (4, N) array."""
    hidden = np.asarray(hidden, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    lab = np.asarray(labels, dtype=np.int64)
    V = weight.shape[1]
    m = np.full(hidden.shape[0], -np.inf)
    for v0 in range(0, V, v_chunk):
        m = np.maximum(m, logits_chunk(hidden, weight, v0, min(V, v0 + v_chunk), softcap).max(1))
    d = np.zeros(hidden.shape[0])
    s = np.zeros(hidden.shape[0])
    for v0 in range(0, V, v_chunk):
        z = logits_chunk(hidden, weight, v0, min(V, v0 + v_chunk), softcap)
        e = np.exp(z - m[:, None])
        d += e.sum(1)
        s += (e * z).sum(1)
    inside = (lab >= v_offset) & (lab < v_offset + V)
    zy = np.zeros(hidden.shape[0])
    idx = np.nonzero(inside)[0]
    if idx.size:
        zy[idx] = _cap(np.einsum("nh,hn->n", hidden[idx], weight[:, lab[idx] - v_offset]),
                       softcap)
    return np.stack([m, d, s, zy])


def combine_shards(stats, labels, reduction="mean", ignore_index=IGNORE_INDEX, zloss_coef=0.0,
                   v_total=None):
    """Whole-vocabulary loss / entropy / lse / E_p[z] from the (P, 4, N) statistics of P
    shards: M = max_p m_p, D = sum_p d_p exp(m_p - M), S = sum_p s_p exp(m_p - M)
    (the online-softmax merge of Liger-Kernel PR #551's first pass), lse = M + log D,
    E_p[z] = S / D, z_y = sum_p z_y,p."""
    st = np.asarray(stats, dtype=np.float64)
    lab = np.asarray(labels, dtype=np.int64)
    if reduction not in _REDS:
        raise ValueError(f"reduction must be one of {_REDS}")
    M = st[:, 0].max(axis=0)
    scale = np.exp(st[:, 0] - M[None, :])
    D = (st[:, 1] * scale).sum(0)
    S = (st[:, 2] * scale).sum(0)
    zy = st[:, 3].sum(0)
    lse = M + np.log(D)
    ez = S / D
    valid = lab != ignore_index
    if v_total is not None and np.any((lab[valid] < 0) | (lab[valid] >= v_total)):
        raise ValueError("label out of range")
    ce = np.where(valid, lse - zy, 0.0)
    ent = np.where(valid, lse - ez, 0.0)
    loss_tok = ce + np.where(valid, zloss_coef * lse * lse, 0.0)
    n_valid = int(valid.sum())
    if reduction == "none":
        loss, entropy = loss_tok, ent
    elif reduction == "sum":
        loss, entropy = float(loss_tok.sum()), float(ent.sum())
    else:
        loss = float(loss_tok.sum()) / n_valid if n_valid else 0.0
        entropy = float(ent.sum()) / n_valid if n_valid else 0.0
    return dict(loss=loss, entropy=entropy, loss_tok=loss_tok, entropy_tok=ent, lse=lse, ez=ez,
                valid=valid, n_valid=n_valid)
