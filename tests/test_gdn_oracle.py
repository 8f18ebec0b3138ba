"""Pins of the Gated DeltaNet recurrence oracle (CPU).

Each pin checks the oracle against something other than its own formula:
hand-worked values, the reset and pure-decay special cases, the associative
memory that the delta rule reduces to for orthonormal keys, the product of
per-token transition matrices, the chunked (WY) form of the same recurrence,
and incremental against whole-sequence processing (the property the Swiftlet
README lists under "Correctness").
"""
import math

import numpy as np
import pytest
from scipy.linalg import solve_triangular

import synth
from oracle import gdn_oracle as G

EPS = 1e-6


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _bf16_bits(x):
    """float -> bf16 bits for values that are exactly representable."""
    f = np.asarray(x, dtype=np.float32)
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(((bits.astype(np.uint32)) << 16).view(np.float32), f)
    return bits


def _rand(seed, T=6, Hk=1, Hv=1, dk=8, dv=5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hk, dk))
    k = rng.standard_normal((T, Hk, dk))
    v = rng.standard_normal((T, Hv, dv))
    alpha = rng.uniform(0.6, 1.0, (T, Hv))
    beta = rng.uniform(0.0, 1.0, (T, Hv))
    S0 = rng.standard_normal((Hv, dv, dk))
    return q, k, v, alpha, beta, S0


def test_first_token_hand_worked():
    """k = (3, 4, 0, 0): |k|^2 = 25; q = (0, 2, 0, 0): |q|^2 = 4; zero state.
    S_1 = beta v k^T / sqrt(25 + eps); o = S_1 q / sqrt(4 + eps) / sqrt(4)."""
    q = _bf16_bits([[[[0, 2, 0, 0]]]])
    k = _bf16_bits([[[[3, 4, 0, 0]]]])
    v = _bf16_bits([[[[1, -2, 0.5]]]])
    alpha, beta = [[[0.7]]], [[[0.5]]]
    out, S = G.gdn_recurrence(q, k, v, alpha, beta, np.zeros((1, 1, 3, 4)))
    nk = math.sqrt(25 + EPS)
    nq = math.sqrt(4 + EPS)
    for i, vi in enumerate([1.0, -2.0, 0.5]):
        for j, kj in enumerate([3.0, 4.0, 0.0, 0.0]):
            assert S[0, 0, i, j] == pytest.approx(0.5 * vi * kj / nk, rel=1e-15, abs=1e-300)
        # S q^ = 0.5 v_i (4 * 2) / (nk nq 2)
        assert out[0, 0, 0, i] == pytest.approx(0.5 * vi * 8.0 / (nk * nq * 2.0), rel=1e-14)


def test_alpha_zero_forgets_the_state():
    q, k, v, alpha, beta, S0 = _rand(1, T=1)
    alpha[:] = 0.0
    _, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    kh = k[0, 0] / math.sqrt(k[0, 0] @ k[0, 0] + EPS)
    np.testing.assert_allclose(S[0], beta[0, 0] * np.outer(v[0, 0], kh), rtol=1e-13, atol=1e-15)


def test_beta_zero_is_pure_decay():
    q, k, v, alpha, beta, S0 = _rand(2, T=5)
    beta[:] = 0.0
    out, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    g = np.cumprod(alpha[:, 0])
    np.testing.assert_allclose(S[0], g[-1] * S0[0], rtol=1e-13)
    for t in range(5):
        qh = q[t, 0] / math.sqrt(q[t, 0] @ q[t, 0] + EPS) / math.sqrt(q.shape[2])
        np.testing.assert_allclose(out[t, 0], g[t] * (S0[0] @ qh), rtol=1e-12, atol=1e-14)


def test_beta_one_writes_v_at_key():
    """With beta = 1 the updated state maps the key to v, up to eps:
    S_t k^ = (1 - c) alpha S k^ + c v with c = |k^|^2 = |k|^2 / (|k|^2 + eps)."""
    q, k, v, alpha, beta, S0 = _rand(3, T=1)
    beta[:] = 1.0
    _, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    kk = k[0, 0] @ k[0, 0]
    kh = k[0, 0] / math.sqrt(kk + EPS)
    c = kk / (kk + EPS)
    want = (1 - c) * alpha[0, 0] * (S0[0] @ kh) + c * v[0, 0]
    np.testing.assert_allclose(S[0] @ kh, want, rtol=1e-12, atol=1e-13)


def test_orthonormal_keys_give_an_overwriting_memory():
    """alpha = beta = 1 and one-hot keys: column j of the state holds the v of
    the last token whose key was e_j (times 1/sqrt(1+eps)); untouched columns
    keep their initial values."""
    dk, dv, T = 6, 4, 9
    rng = np.random.default_rng(4)
    keys = [2, 0, 2, 5, 0, 2, 3, 3, 0]
    k = np.zeros((T, 1, dk))
    for t, j in enumerate(keys):
        k[t, 0, j] = 1.0
    q = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, dv, dk))
    _, S = G.gdn_sequence(q, k, v, np.ones((T, 1)), np.ones((T, 1)), S0)
    for j in range(dk):
        last = [t for t, kj in enumerate(keys) if kj == j]
        if last:
            np.testing.assert_allclose(S[0][:, j], v[last[-1], 0], rtol=2e-6, atol=2e-6)
        else:
            np.testing.assert_array_equal(S[0][:, j], S0[0][:, j])


def _normalised(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + EPS)


def test_product_of_transition_matrices():
    """S_T = S_0 A_1 ... A_T + sum_t beta_t v_t k^_t^T A_{t+1} ... A_T with
    A_t = alpha_t (I - beta_t k^_t k^_t^T), a non-symmetric S_0."""
    T, dk, dv = 7, 6, 4
    q, k, v, alpha, beta, S0 = _rand(5, T=T, dk=dk, dv=dv)
    _, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    kh = _normalised(k[:, 0])
    A = [alpha[t, 0] * (np.eye(dk) - beta[t, 0] * np.outer(kh[t], kh[t])) for t in range(T)]
    want = S0[0].copy()
    for t in range(T):
        want = want @ A[t]
    for t in range(T):
        term = beta[t, 0] * np.outer(v[t, 0], kh[t])
        for s in range(t + 1, T):
            term = term @ A[s]
        want += term
    np.testing.assert_allclose(S[0], want, rtol=1e-12, atol=1e-12)


def test_chunked_wy_form_equals_the_recurrence():
    """The whole-sequence (chunked) form: with decays g_t = prod_{s<=t} alpha_s,
    the per-token deltas u_t = beta_t (v_t - alpha_t S_{t-1} k^_t) solve the unit
    lower-triangular system u_t + beta_t sum_{s<t} (g_t/g_s)(k^_s.k^_t) u_s
    = beta_t (v_t - g_t S_0 k^_t); then o_t = g_t S_0 q^_t + sum_{s<=t}
    (g_t/g_s)(k^_s.q^_t) u_s and S_C = g_C S_0 + sum_s (g_C/g_s) u_s k^_s^T."""
    T, dk, dv = 10, 8, 6
    q, k, v, alpha, beta, S0 = _rand(6, T=T, dk=dk, dv=dv)
    out, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    kh = _normalised(k[:, 0])
    qh = _normalised(q[:, 0]) / math.sqrt(dk)
    g = np.cumprod(alpha[:, 0])
    b = beta[:, 0]
    ratio = g[:, None] / g[None, :]
    Lm = np.tril(b[:, None] * ratio * (kh @ kh.T), -1) + np.eye(T)
    rhs = b[:, None] * (v[:, 0] - g[:, None] * (kh @ S0[0].T))
    U = solve_triangular(Lm, rhs, lower=True, unit_diagonal=True)
    O = g[:, None] * (qh @ S0[0].T) + np.tril(ratio * (qh @ kh.T)) @ U
    Sc = g[-1] * S0[0] + (U * (g[-1] / g)[:, None]).T @ kh
    np.testing.assert_allclose(out[:, 0], O, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S[0], Sc, rtol=1e-11, atol=1e-11)


def test_incremental_equals_whole_sequence():
    q, k, v, alpha, beta, S0 = _rand(7, T=8, Hk=2, Hv=4)
    out, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    o1, S1 = G.gdn_sequence(q[:3], k[:3], v[:3], alpha[:3], beta[:3], S0)
    o2, S2 = G.gdn_sequence(q[3:], k[3:], v[3:], alpha[3:], beta[3:], S1)
    np.testing.assert_array_equal(np.concatenate([o1, o2]), out)
    np.testing.assert_array_equal(S2, S)


def test_value_heads_share_key_heads_in_consecutive_groups():
    """H_v = 4 value heads over H_k = 2 key heads: value heads 0, 1 read key
    head 0 and 2, 3 read key head 1 (every head run alone must agree)."""
    q, k, v, alpha, beta, S0 = _rand(8, T=4, Hk=2, Hv=4)
    out, S = G.gdn_sequence(q, k, v, alpha, beta, S0)
    for h in range(4):
        j = h // 2
        o1, S1 = G.gdn_sequence(q[:, j:j + 1], k[:, j:j + 1], v[:, h:h + 1],
                                alpha[:, h:h + 1], beta[:, h:h + 1], S0[h:h + 1])
        np.testing.assert_array_equal(o1[:, 0], out[:, h])
        np.testing.assert_array_equal(S1[0], S[h])


def test_output_scales_with_query_norm_only_through_eps():
    """q^ is normalised: scaling q by 4 (exact in bf16) changes o by at most
    the eps term's relative effect."""
    q, k, v, alpha, beta, S0 = _rand(9, T=3)
    o1, _ = G.gdn_sequence(q, k, v, alpha, beta, S0)
    o2, _ = G.gdn_sequence(4 * q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(o1, o2, rtol=1e-5)


def test_batched_entry_matches_per_sequence_runs():
    s = synth.GdnShape(Hk=2, Hv=4, dk=8, dv=8)
    q, k, v, a, b, S0 = synth.gdn_inputs(0, 0, 3, 5, s)
    out, S = G.gdn_recurrence(q, k, v, a, b, S0)
    for i in range(3):
        o1, S1 = G.gdn_sequence(G.bf16_to_f64(q[i]), G.bf16_to_f64(k[i]), G.bf16_to_f64(v[i]),
                                _f64(a[i]), _f64(b[i]), _f64(S0[i]))
        np.testing.assert_array_equal(o1, out[i])
        np.testing.assert_array_equal(S1, S[i])
