"""The oracle's pins are strong enough: each planted mistake fails at least one pin.

Mistakes are planted in the oracle module (on the CPU) through monkeypatching,
then the pin functions of ``test_oracle_pins`` run against the broken oracle.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O
from tests import test_oracle_pins as P

PINS = [
    P.test_nibble_order_hand_worked, P.test_dequant_hand_worked, P.test_dequant_matches_brute_rows,
    P.test_zero_point_code_gives_zero_weight, P.test_silu_closed_forms, P.test_softmax_closed_form,
    P.test_topk_all_equal_rows, P.test_topk_one_ulp_apart, P.test_topk_matches_brute_force_sort,
    P.test_zipf_prior_closed_form, P.test_routing_invariants, P.test_permutation_brute_force,
    P.test_block_matches_pure_python_brute_force, P.test_block_with_prior_matches_brute_force,
    P.test_dense_mixture_at_k_equals_E, P.test_identical_experts_reduce_to_one,
    P.test_zero_routed_experts_leave_the_shared_term, P.test_down_projection_is_linear_in_its_scales,
    P.test_hand_worked_block, P.test_bf16_rounding_hand_worked, P.test_rms_norm_hand_worked,
    P.test_rms_norm_invariants, P.test_residual_rounds_the_block_output_first,
    P.test_stack_of_zero_blocks_keeps_the_residual, P.test_stack_matches_pure_python_brute_force,
    P.test_stack_closed_form_layer,
]


def _unpack_high_first(words, cols):
    w = np.asarray(words, dtype=np.uint32)
    shifts = 4 * (7 - np.arange(8, dtype=np.uint32))
    return ((w[..., None] >> shifts) & np.uint32(0xF)).reshape(w.shape[:-1] + (cols,)).astype(np.int64)


def _dequant_no_bias(q, s, b, group, bits=4):
    codes = O.unpack_int4(q, q.shape[-1] * 8).astype(np.float64)
    return np.repeat(O.bf16_to_f64(s), group, axis=-1) * codes


def _dequant_group_off(q, s, b, group, bits=4):
    codes = O.unpack_int4(q, q.shape[-1] * 8).astype(np.float64)
    sc = np.tile(O.bf16_to_f64(s), group)  # wrong group index (c % ngroups)
    bi = np.tile(O.bf16_to_f64(b), group)
    return sc * codes + bi


def _silu_sign(z):
    return z / (1.0 + np.exp(z))


def _topk_high_index_ties(logit, bound, k, exact):
    E = logit.shape[0]
    vals = [exact(e) for e in range(E)]
    return sorted(range(E), key=lambda e: (-vals[e], -e))[:k]


def _topk_ascending(logit, bound, k, exact):
    return list(np.argsort(logit, kind="stable")[:k])


def _mlp_gate_up_swapped(mats, x):
    Wg, Wu, Wd = mats
    return (O.silu(x @ Wu.T) * (x @ Wg.T)) @ Wd.T


def _mlp_down_transposed(mats, x):
    Wg, Wu, Wd = mats
    h = O.silu(x @ Wg.T) * (x @ Wu.T)
    Wt = Wd.reshape(Wd.shape[1], Wd.shape[0]) if Wd.shape[0] != Wd.shape[1] else Wd.T
    return h @ Wt


def _perm_unstable(topk_idx, E):
    flat = np.asarray(topk_idx).reshape(-1)
    order = np.argsort(-np.arange(flat.size))  # reversed pair order inside segments
    order = sorted(order.tolist(), key=lambda p: flat[p])
    counts = np.bincount(flat, minlength=E)
    return np.array(order, np.int32), np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _route_no_renorm(x_bits, W, k):
    idx, wts, gate, logits = ORIG_ROUTE(x_bits, W, k)
    p = np.array([O.softmax(logits[t])[idx[t]] for t in range(idx.shape[0])])
    return idx, p, gate, logits


def _sigmoid_gate_dropped(z):
    return np.ones_like(np.asarray(z, dtype=np.float64))


def _bf16_truncate(v):
    v = np.asarray(v, dtype=np.float64)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _rms_norm_sum(x_bits, norm_w_bits, eps):
    x = O.bf16_to_f64(x_bits)
    g = np.ones_like(x) if norm_w_bits is None else O.bf16_to_f64(norm_w_bits)
    return O.f64_to_bf16_bits(x / np.sqrt(np.sum(x * x) + eps) * g)


def _rms_norm_no_weight(x_bits, norm_w_bits, eps):
    return ORIG_RMS(x_bits, None, eps)


def _rms_norm_no_eps(x_bits, norm_w_bits, eps):
    return ORIG_RMS(x_bits, norm_w_bits, 0.0)


def _residual_unrounded(x_bits, y):
    return O.f64_to_bf16_bits(O.bf16_to_f64(x_bits) + np.asarray(y, np.float64))


ORIG_ROUTE = O.route
ORIG_RMS = O.rms_norm

MUTATIONS = {
    "nibble order high-first": ("unpack_int4", _unpack_high_first),
    "bias dropped": ("dequantize", _dequant_no_bias),
    "wrong group index": ("dequantize", _dequant_group_off),
    "silu sign": ("silu", _silu_sign),
    "ties to highest index": ("select_topk", _topk_high_index_ties),
    "smallest logits selected": ("select_topk", _topk_ascending),
    "gate/up swapped": ("expert_mlp", _mlp_gate_up_swapped),
    "down transposed": ("expert_mlp", _mlp_down_transposed),
    "unstable permutation": ("permutation", _perm_unstable),
    "no renormalisation": ("route", _route_no_renorm),
    "shared gate dropped": ("sigmoid", _sigmoid_gate_dropped),
    "bf16 by truncation": ("f64_to_bf16_bits", _bf16_truncate),
    "rms over the sum, not the mean": ("rms_norm", _rms_norm_sum),
    "norm weight ignored": ("rms_norm", _rms_norm_no_weight),
    "norm eps dropped": ("rms_norm", _rms_norm_no_eps),
    "residual adds y unrounded": ("residual_add", _residual_unrounded),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch, root):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in PINS:
        try:
            if "root" in pin.__code__.co_varnames[:pin.__code__.co_argcount]:
                pin(root)
            else:
                pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutation {name!r}"
