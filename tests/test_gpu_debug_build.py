"""Ragged parity cases through libflce_debug.so, the FLCE_DEBUG build.

That build checks every TMA box and every epilogue store against the extents of its
array before the access (csrc/flce_check.cuh) and reports a failed check as
FLCE_ERR_BOUNDS.  Every call here runs with validate set, so a bounds failure in any
kernel would raise; the results must also match the fp64 oracle as in the regular
parity tests.  The cases are ragged in every dimension (N, H and V off the tile
grid), with several backward vocabulary chunks, token chunks of the gradient-in-
forward mode, the [V,H] layout with an odd vocabulary, vocabulary shards, and every case
of the seeded random sweeps.
"""
import dataclasses

import pytest
import torch

from linear_cross_entropy_forward_gb300 import _binding as B
from linear_cross_entropy_forward_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_forward_gb300.build import build
    prev = B.use_library(build(debug=True))
    try:
        yield
    finally:
        B.restore_library(prev)


W0 = wl.TINY
RAGGED = dataclasses.replace(W0, name="d1", N=300, H=200, V=1000, reduction="none",
                             grad_mode="normal")
CAPPED = dataclasses.replace(W0, name="d2", N=384, H=256, V=2048, w_std=0.3, softcap=2.0,
                             zloss_coef=1e-3)


def test_two_call_path_ragged_and_chunked(debug_library):
    import test_gpu_parity as tp
    tp.check_parity(RAGGED, 256)
    tp.check_parity(CAPPED, 512)
    tp.check_parity(dataclasses.replace(W0, name="d3", N=1, H=8, V=8, ignore_frac=0.0), 0)


def test_weight_vh_odd_vocabulary(debug_library):
    import test_gpu_parity as tp
    tp.check_parity(dataclasses.replace(W0, name="d4", N=300, H=200, V=1001,
                                        reduction="none", grad_mode="normal"), 256,
                    weight_layout="vh")


def test_gradient_in_forward_token_chunks(debug_library):
    import test_gpu_fused as tf
    tf.check_against_oracle(dataclasses.replace(W0, name="d5", N=1100, H=200, V=1000,
                                                reduction="none", grad_mode="normal"), 512)
    tf.check_against_oracle(dataclasses.replace(W0, name="d6", N=1100, H=200, V=1001,
                                                zloss_coef=1e-3), 512, layout="vh")


def test_vocabulary_shards(debug_library):
    import test_gpu_vocab_parallel as tv
    name, w, cuts, layout = tv.CASES[0]
    tv.test_sequential_shards_match_oracle(name, w, cuts, layout)


def test_random_sweep_under_bounds_checks(debug_library):
    """Every case of the seeded random sweeps (C entry points, vocabulary shardings)
    again, now with every TMA box and epilogue store bounds-checked."""
    import test_gpu_random_sweep as ts
    import test_gpu_vocab_parallel as tv
    for i, (w, o) in enumerate(ts.CASES):
        ts.check_case(i, w, o)
    for i, (w, o) in enumerate(ts.CASES2):
        ts.check_case(1000 + i, w, o)
    for case in tv.RANDOM_CASES:
        tv.check_shards(*case)
