"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names the mistake it is there to catch.  All run on the CPU.
"""
import copy
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import moe_oracle as O
from tests import brute

TINY = synth.WORKLOADS[0]


def _tiny_weights(seed=0, layer=0, shape=None, zipf=None):
    shape = shape or TINY.shape
    return synth.layer_weights(seed, 0, layer, shape, zipf_s=zipf)


def _x(T, H, seed=0, layer=0, step=0):
    return synth.tokens(seed, 0, layer, step, T, H)


def _bf16_bits(v):
    """bf16 bits of a value that is exactly representable in bf16."""
    f = np.array([v], np.float32).view(np.uint32)[0]
    assert f & 0xFFFF == 0, v
    return np.uint16(f >> 16)


# --------------------------------------------------------------------------- dequant
def test_nibble_order_hand_worked(root):
    """Catches a high-nibble-first unpack: words from the golden file."""
    with open(os.path.join(root, "tests", "golden", "dequant_hand_worked.json")) as f:
        g = json.load(f)
    for case in g["unpack"]:
        words = np.array([int(w, 16) for w in case["words"]], np.uint32)[None, :]
        assert O.unpack_int4(words, 8 * words.shape[1])[0].tolist() == case["codes"]


def test_dequant_hand_worked(root):
    """Catches a wrong group index, a dropped bias or scale: literal values."""
    with open(os.path.join(root, "tests", "golden", "dequant_hand_worked.json")) as f:
        g = json.load(f)
    for case in g["dequant"]:
        words = np.array([[int(w, 16) for w in case["words"]]], np.uint32)
        s = np.array([[_bf16_bits(v) for v in case["scales"]]], np.uint16)
        b = np.array([[_bf16_bits(v) for v in case["biases"]]], np.uint16)
        W = O.dequantize(words, s, b, case["group"])
        assert W[0].tolist() == case["w"]


def test_dequant_matches_brute_rows():
    W = _tiny_weights()
    ex = W["experts"]
    D = O.dequantize(ex["down_q"][3], ex["down_s"][3], ex["down_b"][3], TINY.G)
    for r in (0, 17, 255):
        ref = brute.dequant_row(ex["down_q"][3][r].tolist(), ex["down_s"][3][r].tolist(),
                                ex["down_b"][3][r].tolist(), TINY.G)
        assert D[r].tolist() == ref


def test_zero_point_code_gives_zero_weight():
    """With b = -8 s (the generator's recipe) code 8 dequantises to exactly 0."""
    W = _tiny_weights()
    ex = W["experts"]
    q = np.full_like(ex["gate_q"][0], 0x88888888)
    D = O.dequantize(q, ex["gate_s"][0], ex["gate_b"][0], TINY.G)
    assert np.all(D == 0.0)


# --------------------------------------------------------------------------- activations
def test_silu_closed_forms():
    assert O.silu(np.float64(0.0)) == 0.0
    assert O.silu(np.float64(1.0)) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert O.silu(np.float64(-1.0)) == pytest.approx(-0.2689414213699951, rel=1e-15)
    assert O.silu(np.float64(30.0)) == pytest.approx(30.0, rel=1e-12)
    assert abs(O.silu(np.float64(-40.0))) < 1e-15
    assert O.sigmoid(np.float64(0.0)) == 0.5


def test_softmax_closed_form():
    p = O.softmax(np.array([0.0, math.log(3.0)]))
    assert p.tolist() == pytest.approx([0.25, 0.75], rel=1e-15)


# --------------------------------------------------------------------------- routing
def test_exact_logit_is_exact():
    # 1 + 2^-40 - 1: float64 summation in the wrong order would lose the tail
    x = np.array([_bf16_bits(1.0), _bf16_bits(2.0 ** -20), _bf16_bits(-1.0)], np.uint16)
    w = np.array([_bf16_bits(1.0), _bf16_bits(2.0 ** -20), _bf16_bits(1.0)], np.uint16)
    assert O.exact_logit(x, w) == Fraction(1, 2 ** 40)


def test_router_bound_holds():
    W = _tiny_weights()
    x = _x(16, TINY.H)
    logits, bound = O.router_logits(x, W["router_w"])
    for t in range(0, 16, 5):
        for e in range(TINY.E):
            ex = O.exact_logit(x[t], W["router_w"][e])
            assert abs(Fraction(float(logits[t, e])) - ex) <= Fraction(float(bound[t, e]))


def test_topk_all_equal_rows():
    """Identical router rows: ties everywhere -> lowest indices, weights 1/k."""
    W = _tiny_weights()
    W["router_w"] = np.repeat(W["router_w"][:1], TINY.E, axis=0)
    x = _x(3, TINY.H)
    idx, wts, _, _ = O.route(x, W, 5)
    assert idx.tolist() == [[0, 1, 2, 3, 4]] * 3
    assert np.allclose(wts, 0.2, rtol=0, atol=1e-15)


def test_topk_one_ulp_apart():
    """Rows that differ by one bf16 ulp in one weight, probed by a one-hot x."""
    E, H = 6, 32
    rw = np.zeros((E, H), np.uint16)
    base = 0x3F80  # 1.0
    # expert e gets 1.0 + (perm[e]) ulps at column 0 -> known order
    perm = [2, 5, 0, 4, 1, 3]
    for e in range(E):
        rw[e, 0] = base + perm[e]
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = _bf16_bits(1.0)
    W = {"router_w": rw, "router_bias": None, "shared_gate_w": np.zeros(H, np.uint16)}
    idx, _, _, _ = O.route(x, W, 4)
    assert idx[0].tolist() == [1, 3, 5, 0]


def test_topk_matches_brute_force_sort():
    """Catches wrong candidate pruning: full exact sort on tiny E, random and near-tie rows."""
    rng = np.random.default_rng(0)
    W = _tiny_weights()
    x = _x(6, TINY.H)
    rw = W["router_w"].copy()
    # plant exact and near ties: duplicate rows, and rows one ulp apart in one column
    rw[5] = rw[2]
    rw[9] = rw[2]
    rw[7] = rw[11]
    rw[7, 3] ^= 1
    W["router_w"] = rw
    for k in (1, 2, 5, 16):
        idx, _, _, _ = O.route(x, W, k)
        for t in range(x.shape[0]):
            exact = [O.exact_logit(x[t], rw[e]) for e in range(TINY.E)]
            ref = sorted(range(TINY.E), key=lambda e: (-exact[e], e))[:k]
            assert idx[t].tolist() == ref
    # scaled so that many logits tie after float64 rounding
    x2 = np.repeat(x[:1], 2, axis=0)
    idx, _, _, _ = O.route(x2, W, 4)
    assert idx[0].tolist() == idx[1].tolist()
    del rng


def test_zipf_prior_closed_form():
    """x = 0: logits are the prior -s ln(e+1); top-k = 0..k-1 and w_j ~ (j+1)^-s."""
    shape = TINY.shape
    W = _tiny_weights(zipf=1.1)
    x = np.zeros((1, shape.H), np.uint16)
    idx, wts, gate, _ = O.route(x, W, 3)
    assert idx[0].tolist() == [0, 1, 2]
    z = np.array([1.0, 2.0 ** -1.1, 3.0 ** -1.1])
    # the prior is stored in float32: compare at float32 precision
    assert np.allclose(wts[0], z / z.sum(), rtol=1e-6)
    assert gate[0] == 0.5


def test_routing_invariants():
    W = _tiny_weights(zipf=0.8)
    x = _x(32, TINY.H, step=3)
    idx, wts, _, logits = O.route(x, W, 4)
    for t in range(32):
        assert len(set(idx[t].tolist())) == 4
        assert all(logits[t, idx[t, j]] >= logits[t, idx[t, j + 1]] for j in range(3))
        assert abs(wts[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(wts[t]) <= 1e-15)


# --------------------------------------------------------------------------- permutation
def test_permutation_brute_force():
    rng = np.random.default_rng(1)
    for E, T, k in ((16, 4, 2), (8, 50, 3), (512, 7, 10)):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        perm, offsets = O.permutation(idx, E)
        flat = idx.ravel().tolist()
        assert perm.tolist() == sorted(range(T * k), key=lambda p: (flat[p], p))
        assert offsets[0] == 0 and offsets[-1] == T * k
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert all(flat[p] == e for p in seg)
            assert list(seg) == sorted(seg)


# --------------------------------------------------------------------------- whole block
def test_block_matches_pure_python_brute_force():
    """The whole tiny block against an independent pure-Python restatement."""
    W = _tiny_weights()
    x = _x(TINY.T, TINY.H)
    ref = brute.block(x.tolist(), _as_lists(W), TINY.k, TINY.G)
    out = O.moe_block(x, W, TINY.k, TINY.G)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    assert out["perm"].tolist() == ref["perm"]
    assert out["offsets"].tolist() == ref["offsets"]
    assert np.allclose(out["topk_w"], ref["topk_w"], rtol=1e-12, atol=0)
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def test_block_with_prior_matches_brute_force():
    W = _tiny_weights(layer=1, zipf=1.1)
    x = _x(2, TINY.H, layer=1)
    ref = brute.block(x.tolist(), _as_lists(W), 3, TINY.G)
    out = O.moe_block(x, W, 3, TINY.G)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def test_dense_mixture_at_k_equals_E():
    """k = E: y = sum_e softmax_e E_e(x) + g S(x) (no selection, no renormalisation)."""
    W = _tiny_weights()
    x = _x(2, TINY.H)
    out = O.moe_block(x, W, TINY.E, TINY.G)
    for t in range(2):
        xv = [brute.bf16(v) for v in x[t]]
        exact = [float(O.exact_logit(x[t], W["router_w"][e])) for e in range(TINY.E)]
        m = max(exact)
        z = sum(math.exp(v - m) for v in exact)
        y = [0.0] * TINY.H
        for e in range(TINY.E):
            o = brute.mlp(_as_lists(W)["experts"], e, TINY.G, xv)
            pe = math.exp(exact[e] - m) / z
            y = [y[h] + pe * o[h] for h in range(TINY.H)]
        g = 1.0 / (1.0 + math.exp(-sum(a * brute.bf16(b) for a, b in zip(xv, W["shared_gate_w"]))))
        s = brute.mlp(_as_lists(W)["shared"], 0, TINY.G, xv)
        y = np.array([y[h] + g * s[h] for h in range(TINY.H)])
        assert np.max(np.abs(out["y"][t] - y)) <= 1e-12 * np.max(np.abs(y))


def test_identical_experts_reduce_to_one():
    """All experts equal: renormalised weights sum to 1, so y = E_0(x) + g S(x) for any k."""
    W = _tiny_weights()
    for key, v in W["experts"].items():
        W["experts"][key] = np.repeat(v[:1], TINY.E, axis=0)
    x = _x(3, TINY.H)
    X = O.bf16_to_f64(x)
    single = O.expert_mlp(O.expert_matrices(W["experts"], 0, TINY.G), X)
    shared = O.expert_mlp(O.expert_matrices(W["shared"], 0, TINY.G), X)
    gate = O.sigmoid(X @ O.bf16_to_f64(W["shared_gate_w"]))
    for k in (1, 2, 7):
        out = O.moe_block(x, W, k, TINY.G)
        ref = single + gate[:, None] * shared
        assert np.max(np.abs(out["y"] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_zero_routed_experts_leave_the_shared_term():
    """Code 8 everywhere (W = 0): routed terms vanish, y = g S(x) exactly."""
    W = _tiny_weights()
    W["experts"]["gate_q"][:] = 0x88888888
    x = _x(2, TINY.H)
    out = O.moe_block(x, W, TINY.k, TINY.G)
    X = O.bf16_to_f64(x)
    shared = O.expert_mlp(O.expert_matrices(W["shared"], 0, TINY.G), X)
    gate = O.sigmoid(X @ O.bf16_to_f64(W["shared_gate_w"]))
    assert np.array_equal(out["y"], gate[:, None] * shared)


def test_down_projection_is_linear_in_its_scales():
    """Doubling every down scale and bias doubles y exactly (catches a dropped term)."""
    W = _tiny_weights()
    x = _x(2, TINY.H)
    y1 = O.moe_block(x, W, TINY.k, TINY.G)["y"]
    W2 = copy.deepcopy(W)
    for part in ("experts", "shared"):
        for key in ("down_s", "down_b"):
            W2[part][key] = W2[part][key] + np.uint16(0x80)  # +1 in the bf16 exponent = x2
    y2 = O.moe_block(x, W2, TINY.k, TINY.G)["y"]
    assert np.array_equal(y2, 2.0 * y1)


def test_token_independence():
    W = _tiny_weights()
    x = _x(5, TINY.H, step=2)
    full = O.moe_block(x, W, TINY.k, TINY.G)
    for t in range(5):
        one = O.moe_block(x[t:t + 1], W, TINY.k, TINY.G)
        # BLAS may block a batch differently from one row: equal up to rounding
        assert np.allclose(one["y"][0], full["y"][t], rtol=1e-12, atol=1e-14)
        assert one["topk_idx"][0].tolist() == full["topk_idx"][t].tolist()


def test_token_subset():
    W = _tiny_weights()
    x = _x(6, TINY.H)
    full = O.moe_block(x, W, TINY.k, TINY.G)
    sub = O.moe_block(x, W, TINY.k, TINY.G, tokens=[4, 1])
    assert np.allclose(sub["y"], full["y"][[4, 1]], rtol=1e-12, atol=1e-14)


def test_hand_worked_block(root):
    """A block whose output follows in closed form (golden fixture, derivation inside)."""
    with open(os.path.join(root, "tests", "golden", "tiny_block_hand_worked.json")) as f:
        g = json.load(f)
    W, x, k, group = _hand_worked_inputs(g)
    out = O.moe_block(x, W, k, group)
    assert out["topk_idx"].tolist() == g["topk_idx"]
    assert np.allclose(out["topk_w"], g["topk_w"], rtol=1e-12)
    assert np.allclose(out["y"], g["y"], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- helpers
def _as_lists(W):
    def conv(v):
        return None if v is None else v.tolist()
    return {
        "router_w": W["router_w"].tolist(),
        "router_bias": conv(W.get("router_bias")),
        "shared_gate_w": W["shared_gate_w"].tolist(),
        "experts": {k: v.tolist() for k, v in W["experts"].items()},
        "shared": {k: v.tolist() for k, v in W["shared"].items()},
    }


def _hand_worked_inputs(g):
    """Build the fixture's inputs: constant weight matrices W = b (all codes 0)."""
    H, I, E, group = g["H"], g["I"], g["E"], g["group"]

    def const_matrix(rows, cols, value):
        return {"q": np.zeros((rows, cols // 8), np.uint32),
                "s": np.full((rows, cols // group), _bf16_bits(1.0), np.uint16),
                "b": np.full((rows, cols // group), _bf16_bits(value), np.uint16)}

    def expert(cg, cu, cd):
        gm, um, dm = const_matrix(I, H, cg), const_matrix(I, H, cu), const_matrix(H, I, cd)
        return {"gate_q": gm["q"], "gate_s": gm["s"], "gate_b": gm["b"],
                "up_q": um["q"], "up_s": um["s"], "up_b": um["b"],
                "down_q": dm["q"], "down_s": dm["s"], "down_b": dm["b"]}

    exps = [expert(*c) for c in g["experts"]]
    stacked = {key: np.stack([e[key] for e in exps]) for key in exps[0]}
    sh = expert(*g["shared"])
    shared = {key: v[None] for key, v in sh.items()}
    rw = np.array([[_bf16_bits(v) for v in row] for row in g["router_w"]], np.uint16)
    W = {"router_w": rw, "router_bias": None,
         "shared_gate_w": np.array([_bf16_bits(v) for v in g["shared_gate_w"]], np.uint16),
         "experts": stacked, "shared": shared}
    x = np.array([[_bf16_bits(v) for v in row] for row in g["x"]], np.uint16)
    return W, x, g["k"], group


# --------------------------------------------------------------------------- stacks
def test_bf16_rounding_hand_worked():
    """Nearest with ties to even, worked by hand: 1 + 2^-8 is halfway between 1
    and 1 + 2^-7 (even: 1); 1 + 3*2^-8 halfway between 1 + 2^-7 and 1 + 2^-6
    (even: 1 + 2^-6); a hair above a tie rounds up.  Catches truncation and
    ties away from zero."""
    vals = [1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)]
    want = [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81, 0xBF80]
    assert O.f64_to_bf16_bits(np.array(vals)).tolist() == want
    assert [brute.bf16_round(v) for v in vals] == want


def test_rms_norm_hand_worked():
    """x = (3, 4): mean of squares 12.5, x / sqrt(12.5) = (0.84853, 1.13137),
    in bf16 217/256 = 0.84765625 (0x3F59) and 2 * 145/256 = 1.1328125 (0x3F91);
    with g = (2, 0.5): 1.6953125 (0x3FD9) and 0.56640625 (0x3F11)."""
    x = np.array([_bf16_bits(3.0), _bf16_bits(4.0)], np.uint16)
    assert O.rms_norm(x, None, 1e-30).tolist() == [0x3F59, 0x3F91]
    g = np.array([_bf16_bits(2.0), _bf16_bits(0.5)], np.uint16)
    assert O.rms_norm(x, g, 1e-30).tolist() == [0x3FD9, 0x3F11]


def test_rms_norm_invariants():
    """Scaling x by a power of two changes nothing (eps negligible); with unit
    weights the mean square of the output is 1 up to bf16 rounding; eps
    dominates a tiny input: n = x / sqrt(eps)."""
    H = 512
    x = _x(1, H, layer=4)[0]
    n = O.rms_norm(x, None, 1e-30)
    x4 = O.f64_to_bf16_bits(O.bf16_to_f64(x) * 4.0)
    assert np.array_equal(O.rms_norm(x4, None, 1e-30), n)
    ms = float(np.mean(O.bf16_to_f64(n) ** 2))
    assert abs(ms - 1.0) < 2 ** -7
    tiny = O.f64_to_bf16_bits(O.bf16_to_f64(x) * 2.0 ** -40)
    got = O.bf16_to_f64(O.rms_norm(tiny, None, 1.0))
    assert np.allclose(got, O.bf16_to_f64(tiny), rtol=2 ** -7, atol=0)


def test_residual_rounds_the_block_output_first():
    """x = 1, y = 2^-8 + 2^-20: bf16(y) = 2^-8 and 1 + 2^-8 is a tie that goes
    to 1 (even); adding y unrounded would give 1 + 2^-7."""
    x = np.array([_bf16_bits(1.0)], np.uint16)
    assert O.residual_add(x, np.array([2 ** -8 + 2 ** -20])).tolist() == [0x3F80]
    assert O.residual_add(x, np.array([3 * 2 ** -8])).tolist() == [0x3F82]


def test_stack_of_zero_blocks_keeps_the_residual():
    """All expert and shared weights zero: every block outputs 0 and x passes
    through every layer unchanged, whatever the norm weights."""
    W = _tiny_weights(layer=2)
    for part in ("experts", "shared"):
        for m in ("gate", "up", "down"):
            W[part][m + "_q"] = np.zeros_like(W[part][m + "_q"])
            W[part][m + "_b"] = np.zeros_like(W[part][m + "_b"])
    x = _x(1, TINY.H, layer=2)[0]
    g = [O.f64_to_bf16_bits(np.full(TINY.H, 1.5))] * 3
    out = O.moe_stack(x, [W] * 3, g, TINY.k, TINY.G, 1e-6)
    assert np.all(out["y"] == 0.0)
    for l in range(4):
        assert np.array_equal(out["x"][l], x)


def test_stack_matches_pure_python_brute_force():
    """Three tiny layers with their own weights and norm weights against the
    pure-Python restatement (integer bf16 rounding, fsum, exact logits)."""
    Ws = [_tiny_weights(layer=10 + l) for l in range(3)]
    x = _x(1, TINY.H, layer=10)[0]
    rng = np.random.default_rng(5)
    g = [O.f64_to_bf16_bits(1.0 + 0.25 * rng.standard_normal(TINY.H)) for _ in range(3)]
    out = O.moe_stack(x, Ws, g, TINY.k, TINY.G, 1e-6)
    ref = brute.stack(x.tolist(), [_as_lists(W) for W in Ws], [v.tolist() for v in g],
                      TINY.k, TINY.G, 1e-6)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    assert out["xn"].tolist() == ref["xn"]
    assert out["x"].tolist() == ref["x"]
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def test_stack_given_inputs_replace_the_norm():
    """xn_given feeds each block exactly that input (the residual still runs)."""
    Ws = [_tiny_weights(layer=20 + l) for l in range(2)]
    x = _x(1, TINY.H, layer=20)[0]
    xn = _x(2, TINY.H, layer=21)
    out = O.moe_stack(x, Ws, None, TINY.k, TINY.G, 1e-6, xn_given=xn)
    for l in range(2):
        ref = brute.block([xn[l].tolist()], _as_lists(Ws[l]), TINY.k, TINY.G)
        assert out["topk_idx"][l].tolist() == ref["topk_idx"][0]
        assert np.array_equal(out["xn"][l], xn[l])


def test_stack_closed_form_layer():
    """The closed-form layer of the C++ oracle's pins (block output 2^-8 + 2^-20,
    residual tie to even) on the numpy oracle."""
    from tests.test_oracle_cpp import closed_form_stack_layer
    W, x = closed_form_stack_layer()
    out = O.moe_stack(x, [W], None, TINY.k, TINY.G, 1e-6)
    assert np.all(out["xn"][0] == 0x3F80)
    assert np.all(out["y"][0] == 2.0 ** -8 + 2.0 ** -20)
    assert np.all(out["x"][1] == 0x3F80)
