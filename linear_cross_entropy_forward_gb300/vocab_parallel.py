"""Vocabulary-parallel fused linear cross-entropy + entropy.

Each rank holds one slice of the vocabulary (weight columns [v_offset, v_offset + V_r)
of v_total).  The forward needs one exchange: every rank computes the online-softmax
statistics of its slice per token, (m, d, s, z_y) -- the quantities the Liger-Kernel
PR #551 review calls m and d of the first online-softmax pass, plus the centred sum
the entropy needs -- the ranks all-gather them, and each merges the [P, 4, N] block by
max-rescaling into lse, E_p[z], CE and entropy for the whole vocabulary.  The backward
needs one more: each rank's dhidden is its slice's term, summed by an all-reduce;
dweight stays sharded.  The terms are kept in fp32 (the backward's unrounded
accumulation) for the sum, which is rounded to hidden's dtype once, after it.
Labels, hidden and the upstream gradients are replicated.
"""
from __future__ import annotations

import torch

from . import _binding as B
from .workloads import IGNORE_INDEX, RED_NONE, reduction_code


def exchange_stats(local_stats: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather each rank's [4, N] shard statistics into [P, 4, N] (rank order)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return local_stats.unsqueeze(0)
    world = dist.get_world_size(group)
    rows, n = local_stats.shape
    # the concatenated [P*4, N] output form is what every backend accepts
    out = torch.empty(world * rows, n, dtype=local_stats.dtype, device=local_stats.device)
    dist.all_gather_into_tensor(out, local_stats.contiguous(), group=group)
    return out.view(world, rows, n)


def reduce_dhidden(dh_partial: torch.Tensor, group=None) -> torch.Tensor:
    """Sum each rank's dhidden term over the ranks (in fp32, fp64 stays fp64); the
    result has the term's dtype."""
    import torch.distributed as dist
    acc = dh_partial.double() if dh_partial.dtype == torch.float64 else dh_partial.float()
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return acc.to(dh_partial.dtype)


class _VocabParallelCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight_shard, labels, v_offset, v_total, reduction, ignore_index,
                zloss_coef, softcap, weight_layout, group):
        stats = B.flce_shard_stats(hidden, weight_shard, labels, v_offset, v_total, softcap,
                                   ignore_index, weight_layout)
        all_stats = exchange_stats(stats, group)
        loss, ent, lse, ez = B.flce_combine_shards(all_stats, labels, v_total, reduction,
                                                   ignore_index, zloss_coef, H=hidden.shape[1])
        ctx.save_for_backward(hidden, weight_shard, labels, lse, ez)
        ctx.cfg = (v_offset, v_total, reduction, ignore_index, zloss_coef, softcap,
                   weight_layout, group)
        if reduction_code(reduction) != RED_NONE:
            loss, ent = loss[0], ent[0]
        return loss, ent

    @staticmethod
    def backward(ctx, g_loss, g_ent):
        hidden, weight_shard, labels, lse, ez = ctx.saved_tensors
        (v_offset, v_total, reduction, ignore_index, zloss_coef, softcap, weight_layout,
         group) = ctx.cfg
        n_g = hidden.shape[0] if reduction_code(reduction) == RED_NONE else 1

        def prep(g):
            return None if g is None else g.detach().reshape(n_g).float().contiguous()

        dh, dw = B.flce_backward(hidden, weight_shard, labels, lse, ez, prep(g_loss), prep(g_ent),
                                 reduction, ignore_index, zloss_coef, softcap,
                                 weight_layout=weight_layout, v_offset=v_offset,
                                 v_total=v_total, dhidden_fp32=True)
        return (reduce_dhidden(dh, group).to(hidden.dtype), dw, None, None, None, None, None,
                None, None, None, None)


def vocab_parallel_linear_cross_entropy(hidden, weight_shard, labels, v_offset, v_total,
                                        reduction="mean", ignore_index=IGNORE_INDEX,
                                        zloss_coef=0.0, softcap=0.0, weight_layout="hv",
                                        group=None):
    """loss, entropy over the whole vocabulary from this rank's weight slice.

    weight_shard: [H, V_r] ('hv') or [V_r, H] ('vh') bf16, columns [v_offset,
    v_offset + V_r) of v_total.  Collective over `group` (all ranks call it with
    replicated hidden / labels).  Gradients: dhidden summed over ranks, dweight of
    this slice.
    """
    return _VocabParallelCE.apply(hidden, weight_shard, labels, int(v_offset), int(v_total),
                                  reduction, ignore_index, zloss_coef, softcap, weight_layout,
                                  group)
