"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Every mutation patches one oracle function for the duration of one pin; the
pin must then fail.  This shows the pins are strong enough to catch a dropped
term, a swapped operand, a wrong sign or index, a lost temperature factor.
"""
import numpy as np
import pytest

from oracle import kd_oracle as O
from tests import test_oracle_pins as P


def _swap_pq_forward(orig):
    def kl_rows(a_s, a_t, variant, beta=0.5):
        if variant == "forward":
            return orig(a_t, a_s, variant, beta)
        return orig(a_s, a_t, variant, beta)
    return kl_rows


def _drop_reverse_baseline(orig):
    def kl_grad_rows(variant, aux, beta=0.5):
        if variant == "reverse":
            return aux["p"] * (aux["logp"] - aux["logq"])
        return orig(variant, aux, beta)
    return kl_grad_rows


def _skew_weights_swapped(orig):
    def kl_rows(a_s, a_t, variant, beta=0.5):
        return orig(a_s, a_t, variant, 1.0 - beta if variant.startswith("skew") else beta)
    return kl_rows


def _label_off_by_one(orig):
    def ce(z, labels, valid):
        return orig(z, np.minimum(np.asarray(labels) + 1, z.shape[1] - 1), valid)
    return ce


def _transposed_dw(orig):
    def hidden_grads(h_s, w_s, g_s, h_t=None, g_t=None, tied=False):
        d_h, d_w = orig(h_s, w_s, g_s, h_t, g_t, tied)
        return d_h, d_w[::-1].copy()
    return hidden_grads


def _topk_renormalised(orig):
    def topk_rows(a, idx, pk):
        pk = O.as_f64(pk)
        return orig(a, idx, pk / pk.sum(axis=-1, keepdims=True))
    return topk_rows


def _temper_after_aggregation(orig):
    def project_teacher_logits(z_t, token_map, v_student, temperature=1.0):
        return orig(z_t, token_map, v_student, 1.0) / temperature
    return project_teacher_logits


def _unmatched_get_zero_logit(orig):
    def project_teacher_logits(z_t, token_map, v_student, temperature=1.0):
        out = orig(z_t, token_map, v_student, temperature)
        out[np.isneginf(out)] = 0.0
        return out
    return project_teacher_logits


def _mix_logits_not_probabilities(orig):
    def mix_teacher_logits(logits, weights=None, mode="arithmetic"):
        return orig(logits, weights, "geometric")  # a weighted sum of log-probabilities
    return mix_teacher_logits


def _mix_weights_unnormalised(orig):
    def mix_teacher_logits(logits, weights=None, mode="arithmetic"):
        w = np.ones(len(logits)) if weights is None else np.asarray(weights, dtype=np.float64)
        return orig(logits, w, mode) + (np.log(w.sum()) if mode == "arithmetic" else 0.0)
    return mix_teacher_logits


def _geometric_not_renormalised(orig):
    def mix_teacher_logits(logits, weights=None, mode="arithmetic"):
        out = orig(logits, weights, mode)
        if mode == "geometric":
            w = np.ones(len(logits)) if weights is None else np.asarray(weights, dtype=np.float64)
            w = w / w.sum()
            out = sum(w[k] * O.log_softmax(O.as_f64(z)) for k, z in enumerate(logits))
        return out
    return mix_teacher_logits


def _teacher_dw_sign(orig):
    def teacher_hidden_grads(h_t, w_t, g_t):
        d_h, d_w = orig(h_t, w_t, g_t)
        return d_h, -d_w
    return teacher_hidden_grads


def _no_t_squared():
    orig = O.forward

    def forward(*a, **kw):
        t = kw.get("t_student", 1.0)
        out = orig(*a, **kw)
        if kw.get("w_kl", 1.0) and t != 1.0:
            out["loss"] = out["loss"] / (t * t)
        return out
    return forward


MUTATIONS = [
    ("kl_rows", _swap_pq_forward, lambda: P.test_forward_reverse_kl_match_scipy_entropy(1.0)),
    ("kl_grad_rows", _drop_reverse_baseline,
     lambda: P.test_finite_difference_gradients("separate", "reverse")),
    ("kl_rows", _skew_weights_swapped, lambda: P.test_skew_variants_match_scipy(0.1)),
    ("cross_entropy_rows", _label_off_by_one, P.test_ce_matches_torch_cross_entropy),
    ("hidden_grads", _transposed_dw, lambda: P.test_finite_difference_gradients("tied", "forward")),
    ("topk_rows", _topk_renormalised, P.test_golden_closed_forms),
    ("project_teacher_logits", _temper_after_aggregation,
     P.test_projection_moves_teacher_probability_mass),
    ("project_teacher_logits", _unmatched_get_zero_logit,
     P.test_projection_moves_teacher_probability_mass),
    ("mix_teacher_logits", _mix_logits_not_probabilities, P.test_mix_hand_worked_example),
    ("mix_teacher_logits", _mix_weights_unnormalised, P.test_mix_hand_worked_example),
    ("mix_teacher_logits", _geometric_not_renormalised, P.test_mix_brute_force_probabilities),
    ("teacher_hidden_grads", _teacher_dw_sign,
     lambda: P.test_teacher_gradients_finite_differences("separate", "forward")),
]


@pytest.mark.parametrize("name,mut,pin", MUTATIONS, ids=[m[1].__name__ for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, mut, pin):
    pin()  # the clean oracle passes
    monkeypatch.setattr(O, name, mut(getattr(O, name)))
    with pytest.raises(AssertionError):
        pin()


def test_pin_catches_dropped_t_squared(monkeypatch):
    P.test_t_squared_scaling_and_raw_per_token_kl()
    monkeypatch.setattr(O, "forward", _no_t_squared())
    with pytest.raises(AssertionError):
        P.test_t_squared_scaling_and_raw_per_token_kl()
