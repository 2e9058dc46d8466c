"""fp64 CPU oracle for fused linear cross-entropy + entropy.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.
"""
from .flce_oracle import (IGNORE_INDEX, backward, bf16_bits_to_f64, combine_shards,  # noqa: F401
                          dlogits_chunk, forward, grad_scales, label_logits, logits_chunk,
                          objective, row_stats, shard_stats)
