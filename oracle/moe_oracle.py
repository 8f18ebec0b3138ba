"""CPU oracle of the sparse int4 MoE block -- TEST INFRASTRUCTURE ONLY.

This module is the slow, plain reference that the CUDA library is checked
against.  Only the test suite, the package smoke check and the benchmark's
CPU-baseline leg may import it; the library never does, and it shares no
code with the library (the seeded input generator is the only common module).

What it computes follows the Swiftlet project README ("Show HN: Run an 80B
Qwen in 4.3 GB of RAM on a Mac and a 35B on an iPhone", wpnews), section "How
it works": every token of a layer is routed to k of E experts (8 of 256 for
Qwen3.6-35B-A3B, 10 of 512 for Qwen3-Next-80B-A3B), a shared expert is kept
resident, and the experts are stored in "MLX affine int4/int8 group
quantization" (same README, list of what was built from scratch).  The
block, step by step, is the Qwen3-Next sparse MoE block:

  1. router logits      l[t,e] = x_t . Wr_e (+ prior_e)
  2. softmax over E, top-k (descending, ties -> lowest expert index),
     renormalise the k probabilities to sum to one
  3. shared gate        g_t = sigmoid(x_t . wsg)
  4. token->expert permutation: stable counting sort of the pairs p = t*k + j
  5. per pair           a = Wg x, u = Wu x, h = silu(a) * u, o = Wd h, with
                        W = s*q + b per group of G along the input dimension
  6. combine            y_t = sum_j w_tj o_tj + g_t * S(x_t), S = shared expert

Readings where the sources are silent are marked "Reading:" below.

Precision: every floating-point step runs in float64 (bf16 and fp32 inputs
widen exactly).  Expert selection ranks the *exact* real logits: the float64
value is used where its rounding-error bound certifies the order, and exact
rational arithmetic (``fractions.Fraction``) decides the rest, so the
selection is a function of the inputs alone, not of any summation order.

Parity status: every function here is pinned by the CPU tests (brute force,
closed forms, invariants and hand-worked values); none is "parity unpinned".
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

U64 = 2.0 ** -53  # unit roundoff of float64


# ----------------------------------------------------------------------------
# storage types
# ----------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# MLX affine int4 / int8 group quantisation (Swiftlet README, its list of what
# was built)
# ----------------------------------------------------------------------------
def unpack_int4(words: np.ndarray, cols: int) -> np.ndarray:
    """Codes [rows, cols] from packed words [rows, cols/8].

    Reading: code 8c+j of a row sits in bits 4j..4j+3 of word c (low nibble
    first), the MLX convention for 4-bit packing into uint32.
    """
    w = np.asarray(words, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    codes = (w[..., None] >> shifts) & np.uint32(0xF)
    return codes.reshape(w.shape[:-1] + (cols,)).astype(np.int64)


def unpack_int8(words: np.ndarray, cols: int) -> np.ndarray:
    """Codes [rows, cols] from packed words [rows, cols/4].

    Reading: code 4c+j of a row sits in bits 8j..8j+7 of word c (low byte
    first), the same MLX convention at 8 bits per code.
    """
    w = np.asarray(words, dtype=np.uint32)
    shifts = (8 * np.arange(4, dtype=np.uint32))
    codes = (w[..., None] >> shifts) & np.uint32(0xFF)
    return codes.reshape(w.shape[:-1] + (cols,)).astype(np.int64)


def dequantize(q: np.ndarray, s: np.ndarray, b: np.ndarray, group: int,
               bits: int = 4) -> np.ndarray:
    """W[r, c] = s[r, c // group] * q[r, c] + b[r, c // group]  (float64).

    Reading: groups run along the input (column) dimension; scale and bias are
    bf16 arrays [rows, cols/group]; `bits` is the code width (4 or 8).
    """
    cols = q.shape[-1] * (32 // bits)
    codes = (unpack_int4(q, cols) if bits == 4 else unpack_int8(q, cols)).astype(np.float64)
    sc = np.repeat(bf16_to_f64(s), group, axis=-1)
    bi = np.repeat(bf16_to_f64(b), group, axis=-1)
    return sc * codes + bi


# ----------------------------------------------------------------------------
# router, softmax, exact top-k, renormalisation
# ----------------------------------------------------------------------------
def router_logits(x_bits: np.ndarray, router_w_bits: np.ndarray, router_bias=None):
    """Float64 logits [T, E] and a rigorous bound on their rounding error.

    Every product of two bf16 numbers is exact in float64; a sum of n terms in
    any order is within gamma_n * sum|term| of the exact sum (Higham,
    "Accuracy and Stability of Numerical Algorithms", Thm. 4.3).  The bound
    used is 2*(H+2)*u*(sum|x*w| + |bias|), a factor 2 above that.
    """
    X = bf16_to_f64(x_bits)
    W = bf16_to_f64(router_w_bits)
    logits = X @ W.T
    mag = np.abs(X) @ np.abs(W).T
    if router_bias is not None:
        bvec = f32_to_f64(router_bias)
        logits = logits + bvec[None, :]
        mag = mag + np.abs(bvec)[None, :]
    H = X.shape[1]
    bound = 2.0 * (H + 2) * U64 * mag
    return logits, bound


def exact_logit(x_row_bits, w_row_bits, bias_value=None) -> Fraction:
    """The exact rational value of x . w (+ bias), via fractions.Fraction."""
    xs = bf16_to_f64(x_row_bits)
    ws = bf16_to_f64(w_row_bits)
    total = Fraction(0)
    for xv, wv in zip(xs.tolist(), ws.tolist()):
        if xv != 0.0 and wv != 0.0:
            total += Fraction(xv) * Fraction(wv)
    if bias_value is not None:
        total += Fraction(float(np.float32(bias_value)))
    return total


def select_topk(logit: np.ndarray, bound: np.ndarray, k: int, exact) -> list:
    """The k experts with the largest exact logits, descending; ties -> lowest index.

    ``logit``/``bound``: float64 values and their error bounds for one token;
    ``exact(e)``: the exact value of expert e's logit (a Fraction).

    An expert whose upper bound lies below the k-th largest lower bound is
    beaten by k experts and drops out.  Among the remaining candidates, an
    expert whose interval overlaps another candidate's takes its exact value;
    the others keep the float64 value, which is already ordered correctly
    against every candidate it does not overlap.
    """
    E = logit.shape[0]
    lower = logit - bound
    upper = logit + bound
    kth_lower = np.sort(lower)[E - k]
    cand = [e for e in range(E) if upper[e] >= kth_lower]
    value = {}
    for e in cand:
        overlaps = any(f != e and lower[e] <= upper[f] and lower[f] <= upper[e] for f in cand)
        value[e] = exact(e) if overlaps else float(logit[e])
    # Python compares Fraction and float exactly.
    order = sorted(cand, key=lambda e: (-value[e], e))
    return order[:k]


def softmax(logit: np.ndarray) -> np.ndarray:
    """Plain max-subtracted softmax over all E experts (float64)."""
    m = np.max(logit)
    e = np.exp(logit - m)
    return e / np.sum(e)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    """silu(z) = z * sigmoid(z) = z / (1 + e^-z)."""
    return z / (1.0 + np.exp(-z))


def route(x_bits: np.ndarray, W: dict, k: int):
    """Steps 1-3 for every token.

    Returns (topk_idx int32 [T,k], topk_w float64 [T,k], shared_gate float64 [T],
    logits float64 [T,E]).
    Reading: the renormalisation divides the k selected softmax probabilities
    by their sum, for every k (at k = E it leaves the softmax unchanged).
    """
    x_bits = np.asarray(x_bits)
    T = x_bits.shape[0]
    rw = W["router_w"]
    rb = W.get("router_bias")
    logits, bound = router_logits(x_bits, rw, rb)
    idx = np.zeros((T, k), np.int32)
    wts = np.zeros((T, k), np.float64)
    for t in range(T):
        def exact(e, t=t):
            return exact_logit(x_bits[t], rw[e], None if rb is None else rb[e])
        sel = select_topk(logits[t], bound[t], k, exact)
        p = softmax(logits[t])
        ps = p[sel]
        idx[t] = sel
        wts[t] = ps / np.sum(ps)
    X = bf16_to_f64(x_bits)
    gate = sigmoid(X @ bf16_to_f64(W["shared_gate_w"]))
    return idx, wts, gate, logits


# ----------------------------------------------------------------------------
# permutation
# ----------------------------------------------------------------------------
def permutation(topk_idx: np.ndarray, E: int):
    """Stable counting sort of the pairs p = t*k + j by expert id.

    Returns (perm int32 [T*k], offsets int32 [E+1]): expert e's pairs are
    perm[offsets[e]:offsets[e+1]], in ascending p.
    """
    flat = np.asarray(topk_idx).reshape(-1)
    counts = [0] * E
    for e in flat.tolist():
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:E]
    fill = list(fill)
    perm = [0] * len(flat)
    for p, e in enumerate(flat.tolist()):
        perm[fill[e]] = p
        fill[e] += 1
    return np.array(perm, np.int32), np.array(offsets, np.int32)


# ----------------------------------------------------------------------------
# experts and combine
# ----------------------------------------------------------------------------
def expert_matrices(ex: dict, i: int, group: int, bits: int = 4):
    """Dequantised (Wg [I,H], Wu [I,H], Wd [H,I]) of expert i of a stacked dict."""
    Wg = dequantize(ex["gate_q"][i], ex["gate_s"][i], ex["gate_b"][i], group, bits)
    Wu = dequantize(ex["up_q"][i], ex["up_s"][i], ex["up_b"][i], group, bits)
    Wd = dequantize(ex["down_q"][i], ex["down_s"][i], ex["down_b"][i], group, bits)
    return Wg, Wu, Wd


def expert_mlp(mats, x: np.ndarray) -> np.ndarray:
    """o = Wd (silu(Wg x) * (Wu x)) for x [n, H] (rows independent).

    Reading: SwiGLU applies silu to the gate projection and multiplies by the
    up projection.
    """
    Wg, Wu, Wd = mats
    a = x @ Wg.T
    u = x @ Wu.T
    h = silu(a) * u
    return h @ Wd.T


def moe_block(x_bits: np.ndarray, W: dict, k: int, group: int, tokens=None) -> dict:
    """The whole block.

    ``W``: canonical weights (keys router_w, router_bias, shared_gate_w,
    shared, experts; optional ``bits``, the experts' code width, 4 when
    absent).  ``tokens``: optional list of token rows for which y is computed
    (routing and the permutation always cover every token).

    Returns a dict with y (float64 [len(tokens), H]), topk_idx, topk_w,
    shared_gate, perm, offsets, logits, tokens.
    """
    x_bits = np.asarray(x_bits)
    T, H = x_bits.shape
    E = W["router_w"].shape[0]
    bits = int(W.get("bits", 4))
    idx, wts, gate, logits = route(x_bits, W, k)
    perm, offsets = permutation(idx, E)
    toks = list(range(T)) if tokens is None else [int(t) for t in tokens]
    X = bf16_to_f64(x_bits[toks])
    # expert outputs o[(row, j)], one dequantisation per distinct expert
    pairs = {}
    for r, t in enumerate(toks):
        for j in range(k):
            pairs.setdefault(int(idx[t, j]), []).append((r, j))
    o = np.zeros((len(toks), k, H))
    for e, lst in pairs.items():
        mats = expert_matrices(W["experts"], e, group, bits)
        rows = [r for r, _ in lst]
        out = expert_mlp(mats, X[rows])
        for n, (r, j) in enumerate(lst):
            o[r, j] = out[n]
    shared = expert_mlp(expert_matrices(W["shared"], 0, group, bits), X)
    y = np.zeros((len(toks), H))
    for r, t in enumerate(toks):
        acc = np.zeros(H)
        for j in range(k):
            acc = acc + wts[t, j] * o[r, j]
        y[r] = acc + gate[t] * shared[r]
    return {"y": y, "topk_idx": idx, "topk_w": wts, "shared_gate": gate, "perm": perm,
            "offsets": offsets, "logits": logits, "tokens": toks}


# ----------------------------------------------------------------------------
# a stack of blocks for one token: RMSNorm in, residual out
# ----------------------------------------------------------------------------
# The pages run the blocks one decoder layer after another (README "Status":
# the decode loop is dispatch bound) but print no equations for what sits
# between them.  Reading: the plain pre-norm residual form of the Qwen3-Next
# decoder, without the attention sub-layer: n = RMSNorm(x) * norm_w,
# x <- x + MoE(n); every tensor passed between steps is bf16.
def f64_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even); uint16 bit patterns.

    A finite v = m * 2^e with 1/2 <= |m| < 1 keeps 8 significant bits:
    rint(m * 2^8) * 2^(e - 8), rint rounding half to even.  Values here are
    far from bf16's overflow and underflow, which are not handled.
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)  # exact in float64 and in float32
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rms_norm(x_bits, norm_w_bits, eps: float) -> np.ndarray:
    """bf16 bits of x / sqrt(mean_h x_h^2 + eps) * g (float64, rounded once).

    g = norm_w (bf16) or all ones when norm_w_bits is None.
    """
    x = bf16_to_f64(x_bits)
    g = np.ones_like(x) if norm_w_bits is None else bf16_to_f64(norm_w_bits)
    r = 1.0 / math.sqrt(float(np.mean(x * x)) + eps)
    return f64_to_bf16_bits(x * r * g)


def residual_add(x_bits, y) -> np.ndarray:
    """bf16 bits of x + bf16(y): the block output is rounded to bf16 first."""
    yb = f64_to_bf16_bits(y)
    return f64_to_bf16_bits(bf16_to_f64(x_bits) + bf16_to_f64(yb))


def moe_stack(x_bits, Ws: list, norm_ws, k: int, group: int, eps: float, xn_given=None) -> dict:
    """One token through len(Ws) blocks.

    For l = 0, 1, ...: n_l = rms_norm(x_l), block l on n_l, x_{l+1} =
    residual_add(x_l, y_l).  ``xn_given`` (optional [L][H] bf16 bits)
    replaces each n_l, so that each block can be checked on exactly the input
    another implementation used.  Returns x (inputs, [L+1][H] bits, last =
    the result), xn [L][H] bits, y float64 [L][H], topk_idx [L][k], topk_w.
    """
    x = np.asarray(x_bits, dtype=np.uint16).reshape(-1)
    L = len(Ws)
    xs, xns, ys, idxs, wts = [x], [], [], [], []
    for l in range(L):
        g = None if norm_ws is None else norm_ws[l]
        n = rms_norm(x, g, eps) if xn_given is None else np.asarray(xn_given[l], np.uint16)
        r = moe_block(n[None, :], Ws[l], k, group)
        x = residual_add(x, r["y"][0])
        xns.append(n)
        ys.append(r["y"][0])
        idxs.append(r["topk_idx"][0])
        wts.append(r["topk_w"][0])
        xs.append(x)
    return {"x": np.stack(xs), "xn": np.stack(xns), "y": np.stack(ys),
            "topk_idx": np.stack(idxs), "topk_w": np.stack(wts)}
