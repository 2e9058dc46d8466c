"""Planted mistakes in the oracle must each fail one of its pins.

Each mutant is the oracle's source with one plausible error written in: a dropped
term or factor, a flipped sign, a wrong index, offset or denominator, a missing mask.
The text is executed as a separate module and the pins of test_oracle_pins run
against it (closed forms, worked examples, textbook routines, invariants, finite
differences, the scalar-loop brute force). Every mutant must fail at least one pin,
and the unmodified source must pass all of them. Together these show that the pins
tell a wrong oracle from a right one. Everything runs on the CPU.
"""
import os
import types

import pytest

import test_oracle_pins as pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "flce_oracle.py")

# (name, text in the oracle, replacement): each text occurs exactly once
MUTANTS = [
    ("bf16_shift", "<< np.uint32(16)", "<< np.uint32(15)"),
    ("softcap_drops_c", "return softcap * np.tanh(zp / softcap)", "return np.tanh(zp / softcap)"),
    ("softcap_inner_scale", "return softcap * np.tanh(zp / softcap)",
     "return softcap * np.tanh(zp / (2.0 * softcap))"),
    ("lse_drops_max", "lse = m + np.log(d)", "lse = np.log(d)"),
    ("ez_centred_sum_not_restored", "s += (e * z).sum(axis=1)",
     "s += (e * (z - m[:, None])).sum(axis=1)"),
    ("label_logit_off_by_one", "weight[:, labels[idx]])",
     "weight[:, (labels[idx] + 1) % weight.shape[1]])"),
    ("entropy_sign", "ent = np.where(valid, lse - ez, 0.0)\n    zl =",
     "ent = np.where(valid, ez - lse, 0.0)\n    zl ="),
    ("entropy_not_masked", "ent = np.where(valid, lse - ez, 0.0)\n    zl =",
     "ent = lse - ez\n    zl ="),
    ("zloss_linear", "zloss_coef * lse * lse, 0.0)\n    loss_tok = ce + zl",
     "zloss_coef * lse, 0.0)\n    loss_tok = ce + zl"),
    ("zloss_not_masked", "zl = np.where(valid, zloss_coef * lse * lse, 0.0)",
     "zl = zloss_coef * lse * lse"),
    ("smoothing_over_v_minus_1", "(eps / V) * (cw.sum() * lse - sw)",
     "(eps / (V - 1)) * (cw.sum() * lse - sw)"),
    ("label_class_weight_ignored", "wy = np.where(valid, cw[np.where(valid, lab, 0)], 0.0)",
     "wy = np.where(valid, 1.0, 0.0)"),
    ("mean_ce_over_all_rows", "(float(ce.sum()) / w_valid if w_valid != 0 else 0.0)",
     "(float(ce.sum()) / N)"),
    ("mean_entropy_over_all_rows", "entropy = float(ent.sum()) / n_valid if n_valid > 0 else 0.0",
     "entropy = float(ent.sum()) / N"),
    ("grad_mean_ce_unscaled", "gc *= 1.0 / wv if wv != 0 else 0.0", "gc *= 1.0"),
    ("grad_ignored_entropy_kept", "ge[~valid] = 0.0", "pass"),
    ("grad_zloss_factor_2_dropped", "gl[:, None] * 2.0 * zloss_coef", "gl[:, None] * zloss_coef"),
    ("grad_entropy_sign", "- ge[:, None] * p * (z - ez[:, None])",
     "+ ge[:, None] * p * (z - ez[:, None])"),
    ("grad_entropy_uncentred", "- ge[:, None] * p * (z - ez[:, None])", "- ge[:, None] * p * z"),
    ("grad_softcap_chain_linear", "dz = dz * (1.0 - (z / softcap) ** 2)",
     "dz = dz * (1.0 - z / softcap)"),
    ("grad_softcap_chain_dropped", "dz = dz * (1.0 - (z / softcap) ** 2)", "dz = dz"),
    ("grad_smoothing_term_dropped", "- (eps / V) * cw[v0:v1][None, :]", ""),
    ("grad_onehot_ignores_shard_offset", "np.arange(v_offset + v0, v_offset + v1)",
     "np.arange(v0, v1)"),
    ("dweight_wrong_chunk", "dw[:, v0:v1] = hidden.T @ dz", "dw[:, v0:v1] = hidden.T @ dz[::-1]"),
    ("shard_merge_rescale_sign", "scale = np.exp(st[:, 0] - M[None, :])",
     "scale = np.exp(M[None, :] - st[:, 0])"),
    ("shard_label_boundary", "inside = (lab >= v_offset) & (lab < v_offset + V)",
     "inside = (lab > v_offset) & (lab < v_offset + V)"),
    ("shard_ez_not_rescaled", "S = (st[:, 2] * scale).sum(0)", "S = st[:, 2].sum(0)"),
]

_CASES = pins.json.load(open(pins.GOLDEN))["cases"]

# (label, pin, arguments): cheap pins first; a mutant stops at its first failing pin
PIN_SUITE = (
    [("bf16", pins.test_bf16_widening_is_exact_for_every_bit_pattern, ())]
    + [(f"worked:{c['name']}", pins.test_worked_examples, (c,)) for c in _CASES]
    + [("zero_weight", pins.test_zero_weight_closed_form, args)
       for args in (("none", 0.0, 0.0), ("mean", 0.05, 5.0), ("sum", 0.05, 0.0))]
    + [("single_class", pins.test_single_class, (0.1,)),
       ("all_ignored", pins.test_all_ignored_mean_is_zero, ())]
    + [("torch_ce", pins.test_matches_torch_cross_entropy_and_logsumexp, (r,))
       for r in pins.REDS]
    + [("zloss", pins.test_zloss_adds_coef_lse_squared, ()),
       ("bounds", pins.test_entropy_and_ce_bounds, (2.0,)),
       ("softcap_bounds", pins.test_softcap_bounds_and_large_cap_limit, ()),
       ("shift", pins.test_shift_invariance, ()),
       ("rows_sum", pins.test_dlogit_rows_sum, (0.0,))]
    + [("torch_smoothing", pins.test_smoothing_and_class_weights_match_torch, args)
       for args in (("mean", 0.1, True), ("none", 0.1, False), ("sum", 0.0, True))]
    + [("uniform_weights", pins.test_uniform_class_weights_scale_out_of_the_mean, ())]
    + [("finite_diff", pins.test_backward_matches_finite_differences, args)
       for args in (("mean", 0.1, 1.5), ("none", 0.1, 1.5), ("sum", 0.0, 0.0))]
    + [("finite_diff_smoothing", pins.test_smoothing_weights_zloss_softcap_finite_differences,
        (r,)) for r in ("mean", "none")]
    + [("scalar_loops", pins.test_oracle_matches_scalar_loops, ("mean", 0.05, 2.0)),
       ("shards", pins.test_shard_merge_equals_whole_vocabulary, ("mean", 2.0)),
       ("shards_none", pins.test_shard_merge_equals_whole_vocabulary, ("none", 0.0))]
)


def _source():
    with open(ORACLE_SRC) as f:
        return f.read()


def _module(src, name):
    mod = types.ModuleType(name)
    mod.__file__ = ORACLE_SRC
    exec(compile(src, f"<{name}>", "exec"), mod.__dict__)
    return mod


def _first_failing_pin(mod, monkeypatch, stop_at_first=True):
    monkeypatch.setattr(pins, "orc", mod)
    failed = []
    for label, pin, args in PIN_SUITE:
        try:
            pin(*args)
        except Exception:  # an assertion, or an error the mistake provokes
            failed.append(label)
            if stop_at_first:
                break
    return failed


def test_mutations_apply_once():
    src = _source()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name
        assert old != new, name


def test_unmodified_oracle_passes_every_pin(monkeypatch):
    failed = _first_failing_pin(_module(_source(), "oracle_unmodified"), monkeypatch,
                                stop_at_first=False)
    assert failed == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new, monkeypatch):
    mutant = _module(_source().replace(old, new), f"oracle_mutant_{name}")
    assert _first_failing_pin(mutant, monkeypatch), f"{name}: every pin passed"
