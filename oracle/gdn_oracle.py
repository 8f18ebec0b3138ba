"""Oracle of the Gated DeltaNet recurrence.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline call it; the library never does.

The pages name the layer type but print no equations: three quarters of the
layers of the Qwen hybrid stack are Gated DeltaNet linear attention, whose
recurrent state has a fixed size instead of a KV cache that grows with the
context (wpnews page, Swiftlet README, "How it works"; creativeainews page,
"How Expert Streaming Works").  The reading taken here is the plainest gated
delta rule with one fixed-size state per value head:

  k^ = k / sqrt(|k|^2 + eps),  q^ = q / sqrt(|q|^2 + eps) / sqrt(d_k)
  S~ = alpha_t S_{t-1}                          (gated decay, alpha in [0, 1])
  S_t = S~ + beta_t (v_t - S~ k^) k^T           (delta rule, beta in [0, 1])
  o_t = S_t q^

S is d_v x d_k per value head; value head h reads key head h // (H_v / H_k).
eps = 1e-6.  alpha and beta arrive as inputs (the projections and gates that
produce them, the short convolution, the output norm and the output projection
belong to the rest of the layer and are out of scope).

Everything runs in float64, token by token, as written above.  Pinned by
hand-worked values, special cases, the transition-matrix product and the
chunked (WY) form in the tests.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def l2_normalise(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    """x / sqrt(sum x^2 + eps) along the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gdn_step(S: np.ndarray, q, k, v, alpha: float, beta: float):
    """One token for one value head: returns (S_t, o_t).  q, k are d_k vectors
    (unnormalised), v a d_v vector, S a d_v x d_k matrix."""
    dk = S.shape[1]
    kh = l2_normalise(k)
    qh = l2_normalise(q) / np.sqrt(dk)
    St = alpha * np.asarray(S, dtype=np.float64)
    St = St + beta * np.outer(np.asarray(v, np.float64) - St @ kh, kh)
    return St, St @ qh


def gdn_sequence(q, k, v, alpha, beta, state):
    """One sequence, float64 arrays: q, k [T][H_k][d_k]; v [T][H_v][d_v];
    alpha, beta [T][H_v]; state [H_v][d_v][d_k] (not modified).
    Returns (out [T][H_v][d_v], state_T)."""
    T, Hk, _ = q.shape
    Hv = v.shape[1]
    group = Hv // Hk
    S = np.array(state, dtype=np.float64, copy=True)
    out = np.zeros((T, Hv, v.shape[2]))
    for t in range(T):
        for h in range(Hv):
            j = h // group
            S[h], out[t, h] = gdn_step(S[h], q[t, j], k[t, j], v[t, h],
                                       float(alpha[t][h]), float(beta[t][h]))
    return out, S


def gdn_recurrence(q_bits, k_bits, v_bits, alpha, beta, state):
    """B independent sequences of T tokens (the kernel's layout).

    q_bits, k_bits: bf16 bits [B][T][H_k][d_k]; v_bits: bf16 bits [B][T][H_v][d_v];
    alpha, beta: float [B][T][H_v]; state: float [B][H_v][d_v][d_k] (not modified).
    Returns (out [B][T][H_v][d_v], state_T [B][H_v][d_v][d_k]), float64.
    """
    q, k, v = bf16_to_f64(q_bits), bf16_to_f64(k_bits), bf16_to_f64(v_bits)
    al = np.asarray(alpha, dtype=np.float64)
    be = np.asarray(beta, dtype=np.float64)
    st = np.asarray(state, dtype=np.float64)
    B = q.shape[0]
    outs, states = [], []
    for b in range(B):
        o, S = gdn_sequence(q[b], k[b], v[b], al[b], be[b], st[b])
        outs.append(o)
        states.append(S)
    return np.stack(outs), np.stack(states)
