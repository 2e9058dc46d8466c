"""The seeded input generators, on the CPU: the workloads' stated recipe (shapes, dtypes,
value distributions, exact ignore counts, upstream gradients, self-sampled labels) and
determinism.  Both the CUDA path and the oracle receive these inputs, so a wrong recipe
would go unnoticed by parity alone."""
import dataclasses
import math

import pytest
import torch

from linear_cross_entropy_forward_gb300 import workloads as wl


def _small(w, N=512, H=64, V=1000):
    return w.scaled(w.name + "_small", N, H, V)


@pytest.mark.parametrize("w", list(wl.WORKLOADS.values()), ids=list(wl.WORKLOADS))
def test_recipe_at_small_size(w):
    s = _small(w)
    hidden, weight, labels, g_loss, g_ent = wl.make_inputs(s)
    assert hidden.shape == (s.N, s.H) and hidden.dtype == torch.bfloat16
    assert weight.shape == (s.H, s.V) and weight.dtype == torch.bfloat16
    assert labels.shape == (s.N,) and labels.dtype == torch.int64
    ign = labels == wl.IGNORE_INDEX
    assert int(ign.sum()) == round(s.ignore_frac * s.N)
    assert bool(((labels[~ign] >= 0) & (labels[~ign] < s.V)).all())
    h = hidden.float()
    assert abs(h.mean().item()) < 0.02 and abs(h.std().item() - 1.0) < 0.02
    assert abs(weight.float().std().item() / s.w_std - 1.0) < 0.02
    n_g = s.N if s.reduction == "none" else 1
    assert g_loss.shape == (n_g,) and g_ent.shape == (n_g,)
    assert g_loss.dtype == torch.float32 and g_ent.dtype == torch.float32
    if s.grad_mode == "ones":
        assert bool((g_loss == 1).all() and (g_ent == 1).all())
    elif s.grad_mode == "normal":
        assert abs(g_loss.std().item() - 1.0) < 0.1 and abs(g_ent.std().item() - 1.0) < 0.1
        assert not torch.equal(g_loss, g_ent)
    else:  # rl: g_loss = 1, g_entropy = the entropy coefficient, per token
        assert bool((g_loss == 1).all())
        assert bool((g_ent == torch.tensor(s.g_ent_coef, dtype=torch.float32)).all())


def test_the_five_shapes():
    shapes = {k: (w.N, w.H, w.V) for k, w in wl.WORKLOADS.items()}
    assert shapes == {"tiny": (256, 512, 4096), "llama2_7b_head": (4096, 4096, 32000),
                      "llama3_8b_head": (8192, 4096, 128256),
                      "gemma2_2b_head_softcap": (4096, 2304, 256000),
                      "qwen25_7b_rl_batch": (16384, 3584, 152064)}
    assert wl.WORKLOADS["llama3_8b_head"].zloss_coef == 1e-4
    assert wl.WORKLOADS["gemma2_2b_head_softcap"].softcap == 30.0
    assert wl.WORKLOADS["gemma2_2b_head_softcap"].w_std == 0.03


def test_deterministic_and_independent_streams():
    s = _small(wl.LLAMA2)
    a = wl.make_inputs(s)
    b = wl.make_inputs(s)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    c = wl.make_inputs(dataclasses.replace(s, seed=1))
    assert not torch.equal(a[0], c[0]) and not torch.equal(a[1], c[1])
    # hidden and weight come from different sub-streams: no shared prefix
    h = a[0].float().flatten()[:64]
    w = (a[1].float() / s.w_std).flatten()[:64]
    assert not torch.allclose(h, w, atol=0.05)


def test_values_are_bf16_rounded_fp32_draws():
    s = _small(wl.TINY)
    h = wl.make_hidden(s)
    ref = torch.randn(s.N, s.H, generator=wl._gen(s.seed)).to(torch.bfloat16)
    assert torch.equal(h.view(torch.int16), ref.view(torch.int16))


def test_self_sampled_labels_follow_the_tempered_softmax():
    """Gumbel-max sampling from softmax(T z): over many rows, the mean probability of the
    sampled label equals the mean of sum_v p_v^2 (its expectation under correct sampling);
    an argmax without noise or the wrong temperature misses it."""
    s = dataclasses.replace(wl.QWEN25, name="q_small", N=20000, H=16, V=50, ignore_frac=0.0,
                            w_std=0.1)
    hidden, weight = wl.make_hidden(s), wl.make_weight(s)
    labels = wl.make_labels(s, hidden, weight)
    z = hidden.float() @ weight.float()
    p = torch.softmax(s.label_temp * z.double(), dim=1)
    got = p[torch.arange(s.N), labels].mean().item()
    expect = (p * p).sum(1).mean().item()
    se = p.max(1).values.std().item() / math.sqrt(s.N)
    assert abs(got - expect) < 5 * se + 1e-3
    # the labels are peaked: far more likely than a uniform draw
    assert got > 3.0 / s.V
