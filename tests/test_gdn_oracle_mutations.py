"""Each mistake planted in the Gated DeltaNet oracle (on the CPU, by
monkeypatching) fails at least one of its pins."""
import numpy as np
import pytest

from oracle import gdn_oracle as G
from tests import test_gdn_oracle as P

PINS = [
    P.test_first_token_hand_worked, P.test_alpha_zero_forgets_the_state,
    P.test_beta_zero_is_pure_decay, P.test_beta_one_writes_v_at_key,
    P.test_orthonormal_keys_give_an_overwriting_memory, P.test_product_of_transition_matrices,
    P.test_chunked_wy_form_equals_the_recurrence, P.test_incremental_equals_whole_sequence,
    P.test_value_heads_share_key_heads_in_consecutive_groups,
    P.test_output_scales_with_query_norm_only_through_eps,
    P.test_batched_entry_matches_per_sequence_runs,
]


def _step(variant):
    def step(S, q, k, v, alpha, beta):
        dk = S.shape[1]
        S = np.asarray(S, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        kh = G.l2_normalise(k) if variant != "raw_k" else np.asarray(k, np.float64)
        qh = G.l2_normalise(q) / np.sqrt(dk)
        if variant == "no_q_scale":
            qh = G.l2_normalise(q)
        if variant == "raw_q":
            qh = np.asarray(q, np.float64) / np.sqrt(dk)
        St = alpha * S
        if variant == "delta_on_old_state":
            St = St + beta * np.outer(v - S @ kh, kh)
        elif variant == "decay_after_update":
            St = alpha * (S + beta * np.outer(v - S @ kh, kh))
        elif variant == "beta_on_v_only":
            St = St + np.outer(beta * v - St @ kh, kh)
        elif variant == "transposed_state":
            St = St + beta * np.outer(v - St.T @ kh, kh) if St.shape[0] == St.shape[1] \
                else St + beta * np.outer(v - (St @ kh)[::-1], kh)
        else:
            St = St + beta * np.outer(v - St @ kh, kh)
        o = St @ qh
        if variant == "output_from_old_state":
            o = (alpha * S) @ qh
        return St, o
    return step


def _norm_eps_outside(x, eps=G.EPS):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)


def _sequence_head_modulo(q, k, v, alpha, beta, state):
    T, Hk, _ = q.shape
    Hv = v.shape[1]
    S = np.array(state, dtype=np.float64, copy=True)
    out = np.zeros((T, Hv, v.shape[2]))
    for t in range(T):
        for h in range(Hv):
            j = h % Hk
            S[h], out[t, h] = G.gdn_step(S[h], q[t, j], k[t, j], v[t, h],
                                         float(alpha[t][h]), float(beta[t][h]))
    return out, S


MUTATIONS = {
    "no_q_scale": ("gdn_step", _step("no_q_scale")),
    "raw_q": ("gdn_step", _step("raw_q")),
    "raw_k": ("gdn_step", _step("raw_k")),
    "delta_on_old_state": ("gdn_step", _step("delta_on_old_state")),
    "decay_after_update": ("gdn_step", _step("decay_after_update")),
    "beta_on_v_only": ("gdn_step", _step("beta_on_v_only")),
    "transposed_state": ("gdn_step", _step("transposed_state")),
    "output_from_old_state": ("gdn_step", _step("output_from_old_state")),
    "eps_outside_sqrt": ("l2_normalise", _norm_eps_outside),
    "head_modulo": ("gdn_sequence", _sequence_head_modulo),
}


def test_unmutated_oracle_passes_every_pin():
    for pin in PINS:
        pin()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(G, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutation {name} passed every pin"
