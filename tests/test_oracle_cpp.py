"""The C++ oracle (oracle/moe_oracle.cpp): pinned on its own, and equal to the
numpy oracle.

The pins below run against any build of the C++ file (``lib``), so that the
mutation test at the end can plant a mistake in a copy of the source, compile
it, and check that some pin fails.  All CPU.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import cpp as C
from oracle import moe_oracle as O
from tests import brute
from tests import test_oracle_pins as P

TINY = synth.WORKLOADS[0]


def _tiny_weights(layer=0, zipf=None, shape=None):
    return synth.layer_weights(0, 0, layer, shape or TINY.shape, zipf_s=zipf)


def _x(T, H, layer=0, step=0):
    return synth.tokens(0, 0, layer, step, T, H)


def _route_only_weights(rw, rb=None):
    """Weights around a given router: tiny zero experts (only routing is read)."""
    E, H = rw.shape
    shape = synth.Shape(E=E, k=1, H=H, I=32, Is=32, G=32)
    W = synth.layer_weights(0, 0, 99, shape)
    W["router_w"] = rw
    W["router_bias"] = rb
    W["shared_gate_w"] = np.zeros(H, np.uint16)
    return W


# ------------------------------------------------------------------- pins
def pin_brute_force_block(lib):
    W = _tiny_weights()
    x = _x(TINY.T, TINY.H)
    ref = brute.block(x.tolist(), P._as_lists(W), TINY.k, TINY.G)
    out = C.moe_block(x, W, TINY.k, TINY.G, lib=lib)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    assert out["perm"].tolist() == ref["perm"]
    assert out["offsets"].tolist() == ref["offsets"]
    assert np.allclose(out["topk_w"], ref["topk_w"], rtol=1e-12, atol=0)
    assert np.allclose(out["shared_gate"], ref["gate"], rtol=1e-12, atol=0)
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def pin_brute_force_block_with_prior(lib):
    W = _tiny_weights(layer=1, zipf=1.1)
    x = _x(2, TINY.H, layer=1)
    ref = brute.block(x.tolist(), P._as_lists(W), 3, TINY.G)
    out = C.moe_block(x, W, 3, TINY.G, lib=lib)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def pin_hand_worked_block(lib, root):
    with open(os.path.join(root, "tests", "golden", "tiny_block_hand_worked.json")) as f:
        g = json.load(f)
    W, x, k, group = P._hand_worked_inputs(g)
    out = C.moe_block(x, W, k, group, lib=lib)
    assert out["topk_idx"].tolist() == g["topk_idx"]
    assert np.allclose(out["topk_w"], g["topk_w"], rtol=1e-12)
    assert np.allclose(out["y"], g["y"], rtol=1e-12, atol=1e-12)


def pin_all_equal_rows(lib):
    """Identical router rows: every logit ties exactly -> lowest ids, weights 1/k."""
    W = _tiny_weights()
    W["router_w"] = np.repeat(W["router_w"][:1], TINY.E, axis=0)
    out = C.moe_block(_x(3, TINY.H), W, 5, TINY.G, lib=lib)
    assert out["topk_idx"].tolist() == [[0, 1, 2, 3, 4]] * 3
    assert np.allclose(out["topk_w"], 0.2, rtol=0, atol=1e-15)


def pin_one_ulp_apart(lib):
    """Expert e's weight at column 0 is 1 + perm[e] bf16 ulps; x is one-hot there."""
    E, H = 6, 32
    rw = np.zeros((E, H), np.uint16)
    order = [2, 5, 0, 4, 1, 3]
    for e in range(E):
        rw[e, 0] = 0x3F80 + order[e]
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80
    out = C.moe_block(x, _route_only_weights(rw), 4, 32, lib=lib)
    assert out["topk_idx"][0].tolist() == [1, 3, 5, 0]


def pin_cancellation_needs_exact_sums(lib):
    """Two rows whose float64 sums differ only through rounding: 2^60 + 1 - 2^60
    against 2^60 - 2^60 + 0.75 (exact values 1 and 0.75)."""
    H = 32
    rw = np.zeros((2, H), np.uint16)
    big = 0x5D80  # bf16 2^60
    rw[0, :3] = [big, 0x3F80, big | 0x8000]          # 2^60, 1, -2^60
    rw[1, :3] = [big, big | 0x8000, 0x3F40]          # 2^60, -2^60, 0.75
    x = np.zeros((1, H), np.uint16)
    x[0, :3] = 0x3F80
    out = C.moe_block(x, _route_only_weights(rw), 1, 32, lib=lib)
    assert out["topk_idx"][0].tolist() == [0]


def pin_dense_mixture(lib):
    """k = E: y = sum_e softmax_e E_e(x) + g S(x), with the experts computed by
    the pure-Python restatement."""
    W = _tiny_weights()
    x = _x(1, TINY.H)
    out = C.moe_block(x, W, TINY.E, TINY.G, lib=lib)
    xv = [brute.bf16(v) for v in x[0]]
    lw = P._as_lists(W)
    logits = [sum(a * brute.bf16(b) for a, b in zip(xv, row)) for row in lw["router_w"]]
    m = max(logits)
    p = [np.exp(v - m) for v in logits]
    p = [v / sum(p) for v in p]
    y = np.zeros(TINY.H)
    for e in range(TINY.E):
        y += p[e] * np.array(brute.mlp(lw["experts"], e, TINY.G, xv))
    g = 1.0 / (1.0 + np.exp(-sum(a * brute.bf16(b) for a, b in zip(xv, lw["shared_gate_w"]))))
    y += g * np.array(brute.mlp(lw["shared"], 0, TINY.G, xv))
    assert np.max(np.abs(out["y"][0] - y)) <= 1e-12 * np.max(np.abs(y))


def pin_stack_brute_force(lib):
    Ws = [_tiny_weights(layer=10 + l) for l in range(3)]
    x = _x(1, TINY.H, layer=10)[0]
    rng = np.random.default_rng(5)
    g = [O.f64_to_bf16_bits(1.0 + 0.25 * rng.standard_normal(TINY.H)) for _ in range(3)]
    out = C.moe_stack(x, Ws, g, TINY.k, TINY.G, 1e-6, lib=lib)
    ref = brute.stack(x.tolist(), [P._as_lists(W) for W in Ws], [v.tolist() for v in g],
                      TINY.k, TINY.G, 1e-6)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    assert out["xn"].tolist() == ref["xn"]
    assert out["x"].tolist() == ref["x"]
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def pin_rms_norm_hand_worked(lib):
    """x = (3, 4) (and zeros), g = (2, 0.5): see the numpy oracle's pin; the
    stack's first normalised input is the RMSNorm alone."""
    H = 256
    x = np.zeros(H, np.uint16)
    x[0], x[1] = 0x4040, 0x4080  # 3, 4
    g = np.full(H, 0x3F80, np.uint16)
    g[0], g[1] = 0x4000, 0x3F00  # 2, 0.5
    # mean of squares 25/256 = (5/16)^2: x * 16/5 * g = (19.2, 6.4) -> bf16 19.25, 6.40625
    out = C.moe_stack(x, [_tiny_weights()], [g], TINY.k, TINY.G, 1e-30, lib=lib)
    assert out["xn"][0][:3].tolist() == [0x419A, 0x40CD, 0]


def closed_form_stack_layer():
    """One layer whose block output is exactly 2^-8 + 2^-20 in every column.

    x = 1 everywhere, so n = RMSNorm(x) = bf16(1 / sqrt(1 + eps)) = 1.  All
    codes are 0, so each matrix is its bias: routed experts 0 (o = 0); shared
    gate 1/4, up 17/16, down 241 * 2^-35; shared-gate vector 0 (g = 1/2).
    a = 256/4 = 64, silu(64) = 64 in float64, u = 272, h = 17408,
    o = 64 * 241 * 2^-35 * 17408 = 4097 * 2^-19, y = o / 2 = 2^-8 + 2^-20.
    Rounded first, bf16(y) = 2^-8 and 1 + 2^-8 is a tie that goes to 1; added
    unrounded, 1 + y rounds to 1 + 2^-7."""
    W = _tiny_weights(layer=3)
    for part in ("experts", "shared"):
        for m in ("gate", "up", "down"):
            W[part][m + "_q"] = np.zeros_like(W[part][m + "_q"])
            W[part][m + "_s"] = np.full_like(W[part][m + "_s"], 0x3F80)
            W[part][m + "_b"] = np.zeros_like(W[part][m + "_b"])
    W["shared"]["gate_b"][:] = 0x3E80   # 0.25
    W["shared"]["up_b"][:] = 0x3F88     # 1.0625
    W["shared"]["down_b"][:] = 0x31F1   # 241 * 2^-35
    W["shared_gate_w"] = np.zeros(TINY.H, np.uint16)
    return W, np.full(TINY.H, 0x3F80, np.uint16)


def pin_residual_rounds_block_output(lib):
    W, x = closed_form_stack_layer()
    out = C.moe_stack(x, [W], None, TINY.k, TINY.G, 1e-6, lib=lib)
    assert np.all(out["xn"][0] == 0x3F80)
    assert np.all(out["y"][0] == 2.0 ** -8 + 2.0 ** -20)
    assert np.all(out["x"][1] == 0x3F80)


def pin_bf16_rounding(lib):
    vals = [1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 1 + 2 ** -8 + 2 ** -20]
    got = np.empty(len(vals), np.uint16)
    v = np.array(vals, np.float64)
    lib.oracle_bf16_round(v.ctypes.data, len(vals), got.ctypes.data)
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]


PINS = [pin_brute_force_block, pin_brute_force_block_with_prior, pin_hand_worked_block,
        pin_all_equal_rows, pin_one_ulp_apart, pin_cancellation_needs_exact_sums,
        pin_dense_mixture, pin_stack_brute_force, pin_rms_norm_hand_worked,
        pin_residual_rounds_block_output, pin_bf16_rounding]


def _run_pin(pin, lib, root):
    if "root" in pin.__code__.co_varnames[:pin.__code__.co_argcount]:
        pin(lib, root)
    else:
        pin(lib)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_cpp_oracle_pin(pin, root):
    _run_pin(pin, C.load(), root)


# ------------------------------------------------------------------- agreement
@pytest.mark.parametrize("case", ["tiny", "prior", "ties", "dense", "35b", "80b", "batched"])
def test_cpp_oracle_equals_numpy_oracle(case):
    wid, T, k = {"tiny": (0, 4, None), "prior": (0, 6, 3), "ties": (0, 3, 4), "dense": (0, 2, 16),
                 "35b": (1, 1, None), "80b": (2, 1, None), "batched": (3, 5, None)}[case]
    wl = synth.WORKLOADS[wid]
    W = synth.layer_weights(0, wl.wid, 2, wl.shape,
                            zipf_s=1.1 if case == "prior" else wl.zipf_s)
    if case == "ties":
        W["router_w"][1::2] = W["router_w"][0::2]  # pairs of equal rows
    k = k or wl.k
    x = synth.tokens(0, wl.wid, 2, 0, T, wl.H)
    a = O.moe_block(x, W, k, wl.G)
    b = C.moe_block(x, W, k, wl.G)
    for key in ("topk_idx", "perm", "offsets"):
        assert np.array_equal(a[key], b[key]), key
    assert np.max(np.abs(a["topk_w"] - b["topk_w"])) <= 1e-14
    assert np.max(np.abs(a["y"] - b["y"])) <= 1e-12 * np.max(np.abs(a["y"]))


def test_cpp_stack_equals_numpy_stack():
    wl = synth.WORKLOADS[1]
    Ws = [synth.layer_weights(0, wl.wid, l, wl.shape) for l in range(2)]
    g = [synth.norm_weights(0, wl.wid, l, wl.H) for l in range(2)]
    x = synth.tokens(0, wl.wid, 0, 0, 1, wl.H)[0]
    a = O.moe_stack(x, Ws, g, wl.k, wl.G, 1e-6)
    b = C.moe_stack(x, Ws, g, wl.k, wl.G, 1e-6)
    for key in ("x", "xn", "topk_idx"):
        assert np.array_equal(a[key], b[key]), key
    assert np.max(np.abs(a["y"] - b["y"])) <= 1e-12 * np.max(np.abs(a["y"]))


def test_cpp_oracle_thread_count_does_not_change_results():
    wl = synth.WORKLOADS[3]
    W = synth.layer_weights(0, wl.wid, 0, wl.shape, zipf_s=wl.zipf_s)
    x = synth.tokens(0, wl.wid, 0, 0, 12, wl.H)
    a = C.moe_block(x, W, wl.k, wl.G, threads=1)
    b = C.moe_block(x, W, wl.k, wl.G, threads=4)
    for key in ("y", "topk_idx", "topk_w", "perm", "offsets"):
        assert np.array_equal(a[key], b[key]), key


# ------------------------------------------------------------------- planted mistakes
MUTATIONS = {
    "nibble order high-first": ("(qr[c / 8] >> (4 * (c % 8)))", "(qr[c / 8] >> (4 * (7 - c % 8)))"),
    "bias dropped": ("* code + bf16_value(br[c / G]);", "* code + 0.0 * bf16_value(br[c / G]);"),
    "wrong group index": ("bf16_value(sr[c / G])", "bf16_value(sr[(c + 1) % m.cols / G])"),
    "ties to the highest id": ("return cand[a] < cand[b];", "return cand[a] > cand[b];"),
    "float64 order only": ("if (need[a] && need[b])", "if (false)"),
    "silu sign": ("return z / (1.0 + std::exp(-z));", "return z / (1.0 + std::exp(z));"),
    "gate/up swapped": ("a[i] = silu(a[i]) * up[i];", "a[i] = silu(up[i]) * a[i];"),
    "no renormalisation": ("for (int j = 0; j < k; ++j) w[j] /= den;", ""),
    "shared gate dropped": ("acc + gate[t] * o[", "acc + 1.0 * o["),
    "unstable permutation": ("for (int p = 0; p < T * k; ++p) perm[fill",
                             "for (int p = T * k - 1; p >= 0; --p) perm[fill"),
    "rms over the sum": ("std::sqrt(ms / H + eps)", "std::sqrt(ms + eps)"),
    "norm weight ignored": ("(norm_w[l] ? bf16_value(norm_w[l][h]) : 1.0)", "1.0"),
    "residual adds y unrounded": ("bf16_value(bf16_round(yl[h]))", "yl[h]"),
    "bf16 by truncation": ("std::nearbyint(std::ldexp(m, 8))", "std::trunc(std::ldexp(m, 8))"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_cpp_mutation_is_caught(name, root, tmp_path):
    old, new = MUTATIONS[name]
    src = open(C.SRC).read()
    assert src.count(old) == 1, f"mutation site of {name!r} not unique"
    mutant = tmp_path / "mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib = C.load(C.build(str(mutant), str(tmp_path / "libmutant.so"), force=True))
    caught = []
    for pin in PINS:
        try:
            _run_pin(pin, lib, root)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutation {name!r}"
