"""Seeded synthetic inputs for fused linear cross-entropy + entropy.

This module only draws random numbers and lays them out. It holds none of the
loss arithmetic: both the CUDA path and the fp64 oracle receive what it makes.

The five workload shapes follow the head shapes the fused-entropy discussion
targets (verl PR #462 "API": bf16 ``hidden [N,H]``, bf16 ``weight [H,V]``,
integer ``labels [N]``), with the feature mix of Liger-Kernel PR #435
(reduction, z-loss) and Liger-Kernel issue #127 (Gemma-2 logit soft-cap).

Seeding: one ``torch.Generator`` per input, seeded ``seed + k`` with
k = 0 hidden, 1 weight, 2 labels, 3 ignore mask, 4 upstream grads,
5 Gumbel noise for self-sampled labels.  Values are drawn in fp32 and rounded
to bf16 (round-to-nearest-even, torch's cast).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

IGNORE_INDEX = -100

RED_NONE, RED_MEAN, RED_SUM = 0, 1, 2
_RED_NAMES = {"none": RED_NONE, "mean": RED_MEAN, "sum": RED_SUM}


def reduction_code(reduction) -> int:
    if isinstance(reduction, int):
        if reduction not in (RED_NONE, RED_MEAN, RED_SUM):
            raise ValueError(f"bad reduction code {reduction}")
        return reduction
    try:
        return _RED_NAMES[reduction]
    except KeyError:
        raise ValueError(f"reduction must be one of none/mean/sum, got {reduction!r}") from None


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    V: int
    w_std: float = 0.02
    ignore_frac: float = 0.1
    reduction: str = "mean"
    zloss_coef: float = 0.0
    softcap: float = 0.0
    # "uniform": labels uniform in [0, V); "self": drawn from softmax(temp * hidden @ weight)
    label_mode: str = "uniform"
    label_temp: float = 4.0
    # upstream gradients: "ones" -> g_loss = g_entropy = 1 (scalar for mean/sum, per token
    # for none); "normal" -> per-token N(0,1) each; "rl" -> g_loss = 1, g_entropy = g_ent_coef
    grad_mode: str = "ones"
    g_ent_coef: float = -0.001
    seed: int = 0

    @property
    def flops_fwd(self) -> float:
        return 2.0 * self.N * self.H * self.V

    @property
    def flops_bwd(self) -> float:
        return 6.0 * self.N * self.H * self.V

    def scaled(self, name: str, N: int, H: int, V: int) -> "Workload":
        """Same recipe at other sizes (parity cases the oracle finishes quickly)."""
        return dataclasses.replace(self, name=name, N=N, H=H, V=V)


# The five shapes: a small case plus four LM-head shapes.
TINY = Workload("tiny", 256, 512, 4096, ignore_frac=0.10, reduction="mean")
LLAMA2 = Workload("llama2_7b_head", 4096, 4096, 32000, ignore_frac=0.05, reduction="none",
                  grad_mode="normal")
LLAMA3 = Workload("llama3_8b_head", 8192, 4096, 128256, ignore_frac=0.20, reduction="mean",
                  zloss_coef=1e-4)
GEMMA2 = Workload("gemma2_2b_head_softcap", 4096, 2304, 256000, w_std=0.03, ignore_frac=0.10,
                  reduction="mean", softcap=30.0)
QWEN25 = Workload("qwen25_7b_rl_batch", 16384, 3584, 152064, ignore_frac=0.15, reduction="none",
                  label_mode="self", label_temp=4.0, grad_mode="rl", g_ent_coef=-0.001)

WORKLOADS = {w.name: w for w in (TINY, LLAMA2, LLAMA3, GEMMA2, QWEN25)}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_hidden(w: Workload) -> torch.Tensor:
    return torch.randn(w.N, w.H, generator=_gen(w.seed + 0)).to(torch.bfloat16)


def make_weight(w: Workload) -> torch.Tensor:
    """``weight [H, V]`` bf16, entries N(0, w_std^2), drawn in row chunks to bound fp32 peak."""
    g = _gen(w.seed + 1)
    out = torch.empty(w.H, w.V, dtype=torch.bfloat16)
    rows = max(1, (1 << 26) // max(1, w.V))
    for r0 in range(0, w.H, rows):
        r1 = min(w.H, r0 + rows)
        out[r0:r1] = (torch.randn(r1 - r0, w.V, generator=g) * w.w_std).to(torch.bfloat16)
    return out


def ignore_rows(w: Workload) -> torch.Tensor:
    """Exactly round(ignore_frac * N) row indices, chosen by a seeded permutation."""
    k = int(round(w.ignore_frac * w.N))
    perm = torch.randperm(w.N, generator=_gen(w.seed + 3))
    return perm[:k]


def _self_sampled_labels(w: Workload, hidden: torch.Tensor, weight: torch.Tensor,
                         device) -> torch.Tensor:
    """Labels drawn from softmax(temp * hidden @ weight) by the Gumbel-max trick.

    This is input preparation, not the loss: it needs the raw scores only to pick
    a token, so it runs plain torch ops (fp32 matmul, CPU or GPU) chunk by chunk.
    """
    dev = torch.device(device)
    g = _gen(w.seed + 5, device=dev)
    h = hidden.to(dev).float()
    best_val = torch.full((w.N,), -math.inf, device=dev)
    best_idx = torch.zeros(w.N, dtype=torch.int64, device=dev)
    chunk = 8192
    for v0 in range(0, w.V, chunk):
        v1 = min(w.V, v0 + chunk)
        s = h @ weight[:, v0:v1].to(dev).float()
        u = torch.rand(w.N, v1 - v0, generator=g, device=dev).clamp_(min=1e-20)
        s.mul_(w.label_temp).sub_(torch.log(-torch.log(u)))
        val, idx = s.max(dim=1)
        upd = val > best_val
        best_val = torch.where(upd, val, best_val)
        best_idx = torch.where(upd, idx + v0, best_idx)
    return best_idx.cpu()


def make_labels(w: Workload, hidden: Optional[torch.Tensor] = None,
                weight: Optional[torch.Tensor] = None, label_device="cpu") -> torch.Tensor:
    if w.label_mode == "uniform":
        labels = torch.randint(0, w.V, (w.N,), generator=_gen(w.seed + 2), dtype=torch.int64)
    elif w.label_mode == "self":
        if hidden is None or weight is None:
            raise ValueError("self-sampled labels need hidden and weight")
        labels = _self_sampled_labels(w, hidden, weight, label_device)
    else:
        raise ValueError(w.label_mode)
    labels[ignore_rows(w)] = IGNORE_INDEX
    return labels


def make_grads(w: Workload):
    """Upstream gradients (g_loss, g_entropy) as fp32 CPU tensors.

    ``reduction='none'`` gives per-token [N] tensors, mean/sum give [1] scalars.
    """
    per_token = w.reduction == "none"
    n = w.N if per_token else 1
    if w.grad_mode == "ones":
        return torch.ones(n), torch.ones(n)
    if w.grad_mode == "normal":
        g = _gen(w.seed + 4)
        return torch.randn(n, generator=g), torch.randn(n, generator=g)
    if w.grad_mode == "rl":
        return torch.ones(n), torch.full((n,), float(w.g_ent_coef))
    raise ValueError(w.grad_mode)


def make_inputs(w: Workload, label_device="cpu"):
    """All inputs of one workload on the CPU: hidden, weight (bf16), labels (int64), grads (fp32)."""
    hidden = make_hidden(w)
    weight = make_weight(w)
    labels = make_labels(w, hidden, weight, label_device=label_device)
    g_loss, g_ent = make_grads(w)
    return hidden, weight, labels, g_loss, g_ent


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns as a numpy uint16 array (exact, for the fp64 oracle)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
