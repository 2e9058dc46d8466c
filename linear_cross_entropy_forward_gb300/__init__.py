"""Fused linear cross-entropy + entropy for NVIDIA GB300 (sm_103a).

loss, entropy = linear_cross_entropy(hidden, weight, labels, reduction="mean")

The [N, V] logits are never materialised: tcgen05 tensor-core GEMM tiles feed
fused online-softmax (forward) and dlogits (backward) epilogues inside
libflce.so, reached through a C ABI (include/flce.h).  The gradient-in-forward
mode (flce_forward_backward, linear_cross_entropy(..., grad_in_forward=True))
keeps one token chunk's logits instead and skips the backward's recompute.
"""
from ._binding import (FlceError, FlceParams, flce_backward, flce_combine_shards,  # noqa: F401
                       flce_forward, flce_forward_backward, flce_scale_bf16,
                       flce_shard_stats, flce_status, kernel_launches,
                       linear_cross_entropy, load_library, make_params, plan_tiles,
                       selftest_wait_timeout, workspace_size,
                       LIB_PATH, EXPORTED)
from .pipeline import HostPipeline  # noqa: F401
from .vocab_parallel import (exchange_stats, reduce_dhidden,  # noqa: F401
                             vocab_parallel_linear_cross_entropy)
from .workloads import IGNORE_INDEX, WORKLOADS  # noqa: F401

__version__ = "0.2.0"
