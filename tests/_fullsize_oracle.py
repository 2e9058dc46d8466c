"""Whole-batch fp64 oracle statistics for the full-size parity tests.

Every row's logsumexp and E_p[z] at a full-size workload cost the oracle a minute or
two of host time (two fp64 passes over all N x V logits).  They depend only on
hidden, weight and the soft-cap, not on the labels, so they are computed once per
process and also kept on disk under tests/.oracle_cache/ (git-ignored), keyed by a
SHA-256 digest of the inputs' bf16 bits, the shapes, the soft-cap and the oracle's own
source (a changed oracle never reads an older entry).  Everything here calls the oracle
only; no value comes from the CUDA path.
"""
from __future__ import annotations

import hashlib
import os

import numpy as np

from oracle import flce_oracle as orc

CACHE_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), ".oracle_cache")
_memo: dict = {}


_ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "flce_oracle.py")


def _digest(h_bits, w_bits, softcap) -> str:
    d = hashlib.sha256()
    with open(_ORACLE_SRC, "rb") as f:
        d.update(f.read())
    for a in (h_bits, w_bits):
        a = np.ascontiguousarray(a)
        d.update(repr((a.shape, a.dtype.str)).encode())
        d.update(memoryview(a).cast("B"))
    d.update(repr(float(softcap)).encode())
    return d.hexdigest()[:40]


def row_stats(h_bits, w_bits, h64, W64, softcap=0.0):
    """orc.row_stats(h64, W64, softcap) for every row: (lse, ez, sw), each [N] fp64.
    h_bits / w_bits are the bf16 bit patterns h64 / W64 were widened from."""
    key = _digest(h_bits, w_bits, softcap)
    if key in _memo:
        return _memo[key]
    path = os.path.join(CACHE_DIR, key + ".npz")
    st = None
    if os.path.exists(path):
        try:
            with np.load(path) as z:
                st = (z["lse"], z["ez"], z["sw"])
            if st[0].shape != (h64.shape[0],):
                st = None
        except (OSError, ValueError, KeyError):
            st = None
    if st is None:
        st = orc.row_stats(h64, W64, softcap)
        os.makedirs(CACHE_DIR, exist_ok=True)
        tmp = path + ".tmp"
        with open(tmp, "wb") as f:
            np.savez(f, lse=st[0], ez=st[1], sw=st[2])
        os.replace(tmp, path)
    _memo[key] = st
    return st


def dweight_columns(V, labels, n=64, seed=7, ignore_index=orc.IGNORE_INDEX):
    """At least `n` vocabulary columns to check dweight on: 16 that are labels of
    non-ignored rows (their one-hot term), 4 in each eighth of the vocabulary (so every
    backward vocabulary chunk of up to eight is hit), the first two and the last
    vocabulary tile of 256 columns (the ragged edge), topped up at random."""
    rng = np.random.default_rng(seed)
    y = np.asarray(labels)
    hit = np.unique(y[y != ignore_index])
    picks = [rng.choice(hit, size=min(16, hit.size), replace=False)] if hit.size else []
    edges = np.linspace(0, V, 9).astype(np.int64)
    for a, b in zip(edges[:-1], edges[1:]):
        if b > a:
            picks.append(rng.integers(a, b, size=min(4, b - a)))
    last0 = max(0, V - 256)
    picks.append(np.array([0, min(1, V - 1), V - 1, max(0, V - 2)]))
    picks.append(rng.integers(last0, V, size=min(4, V - last0)))
    cols = np.unique(np.concatenate(picks))
    while cols.size < min(n, V):
        cols = np.unique(np.concatenate([cols, rng.integers(0, V, size=n - cols.size)]))
    return cols.astype(np.int64)
