"""Pins of the oracle's int8 expert path (CPU), and the mistakes they catch.

The int8 codes follow the same MLX affine convention as the int4 ones at
eight bits per code (Swiftlet README, its list of what was built).
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import moe_oracle as O
from tests import brute

TINY = synth.WORKLOADS[0]


def _bf16_bits(v):
    f = np.array([v], np.float32).view(np.uint32)[0]
    assert f & 0xFFFF == 0, v
    return np.uint16(f >> 16)


def _golden(root):
    with open(os.path.join(root, "tests", "golden", "dequant_hand_worked_int8.json")) as f:
        return json.load(f)


def test_int8_byte_order_hand_worked(root):
    """Catches a high-byte-first unpack or a nibble unpack of int8 words."""
    for case in _golden(root)["unpack"]:
        words = np.array([[int(w, 16) for w in case["words"]]], np.uint32)
        assert O.unpack_int8(words, 4 * words.shape[1])[0].tolist() == case["codes"]


def test_int8_dequant_hand_worked(root):
    """Catches a wrong group index, a dropped scale or bias, or 4-bit columns."""
    for case in _golden(root)["dequant"]:
        words = np.array([[int(w, 16) for w in case["words"]]], np.uint32)
        s = np.array([[_bf16_bits(v) for v in case["scales"]]], np.uint16)
        b = np.array([[_bf16_bits(v) for v in case["biases"]]], np.uint16)
        assert O.dequantize(words, s, b, case["group"], bits=8)[0].tolist() == case["w"]


def test_int8_codes_below_16_equal_int4_codes():
    """The same small codes packed at 8 and at 4 bits dequantise identically."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(5, 64))
    w4 = np.zeros((5, 8), np.uint32)
    w8 = np.zeros((5, 16), np.uint32)
    for r in range(5):
        for c in range(64):
            w4[r, c // 8] |= np.uint32(codes[r, c]) << np.uint32(4 * (c % 8))
            w8[r, c // 4] |= np.uint32(codes[r, c]) << np.uint32(8 * (c % 4))
    s = np.array([[_bf16_bits(0.125), _bf16_bits(-0.5)]] * 5, np.uint16)
    b = np.array([[_bf16_bits(1.0), _bf16_bits(0.25)]] * 5, np.uint16)
    assert np.array_equal(O.dequantize(w4, s, b, 32, bits=4), O.dequantize(w8, s, b, 32, bits=8))


def test_int8_zero_point_and_full_scale():
    """With the generator's b = -128 s: code 128 gives 0, code 0 gives -128 s,
    code 255 gives 127 s, exactly."""
    W = synth.layer_weights_int8(0, 0, 0, TINY.shape)
    ex = W["experts"]
    s = O.bf16_to_f64(ex["gate_s"][0])
    for code, mult in ((0x80, 0.0), (0x00, -128.0), (0xFF, 127.0)):
        q = np.full_like(ex["gate_q"][0], np.uint32(code * 0x01010101))
        D = O.dequantize(q, ex["gate_s"][0], ex["gate_b"][0], TINY.G, bits=8)
        assert np.array_equal(D, np.repeat(mult * s, TINY.G, axis=-1))


def test_int8_dequant_matches_brute_rows():
    W = synth.layer_weights_int8(0, 0, 0, TINY.shape)
    ex = W["experts"]
    D = O.dequantize(ex["down_q"][5], ex["down_s"][5], ex["down_b"][5], TINY.G, bits=8)
    for r in (0, 100, 255):
        ref = brute.dequant_row(ex["down_q"][5][r].tolist(), ex["down_s"][5][r].tolist(),
                                ex["down_b"][5][r].tolist(), TINY.G, bits=8)
        assert D[r].tolist() == ref


def _as_lists(W):
    out = {}
    for k, v in W.items():
        if isinstance(v, dict):
            out[k] = {kk: vv.tolist() for kk, vv in v.items()}
        elif v is None or isinstance(v, int):
            out[k] = v
        else:
            out[k] = v.tolist()
    return out


def test_int8_block_matches_pure_python_brute_force():
    W = synth.layer_weights_int8(0, 0, 2, TINY.shape)
    x = synth.tokens(0, 0, 2, 0, 3, TINY.H)
    ref = brute.block(x.tolist(), _as_lists(W), TINY.k, TINY.G)
    out = O.moe_block(x, W, TINY.k, TINY.G)
    assert out["topk_idx"].tolist() == ref["topk_idx"]
    y = np.array(ref["y"])
    assert np.max(np.abs(out["y"] - y)) <= 1e-12 * np.max(np.abs(y))


def test_int8_block_differs_from_reading_its_words_as_int4():
    """A block that ignored ``bits`` would read the int8 words as int4 codes."""
    W = synth.layer_weights_int8(0, 0, 2, TINY.shape)
    x = synth.tokens(0, 0, 2, 0, 2, TINY.H)
    y8 = O.moe_block(x, W, TINY.k, TINY.G)["y"]
    with pytest.raises(Exception):
        W4 = dict(W)
        W4["bits"] = 4
        O.moe_block(x, W4, TINY.k, TINY.G)  # the int8 words hold twice the columns
    assert np.all(np.isfinite(y8))


# ---- planted mistakes ---------------------------------------------------------

def _pins(root):
    return [lambda: test_int8_byte_order_hand_worked(root),
            lambda: test_int8_dequant_hand_worked(root),
            test_int8_codes_below_16_equal_int4_codes, test_int8_zero_point_and_full_scale,
            test_int8_dequant_matches_brute_rows, test_int8_block_matches_pure_python_brute_force]


def _unpack8_high_first(words, cols):
    w = np.asarray(words, dtype=np.uint32)
    shifts = 8 * (3 - np.arange(4, dtype=np.uint32))
    return ((w[..., None] >> shifts) & np.uint32(0xFF)).reshape(w.shape[:-1] + (cols,)).astype(np.int64)


def _unpack8_seven_bits(words, cols):
    w = np.asarray(words, dtype=np.uint32)
    shifts = 8 * np.arange(4, dtype=np.uint32)
    return ((w[..., None] >> shifts) & np.uint32(0x7F)).reshape(w.shape[:-1] + (cols,)).astype(np.int64)


def _unpack8_signed(words, cols):
    w = np.asarray(words, dtype=np.uint32)
    shifts = 8 * np.arange(4, dtype=np.uint32)
    u = ((w[..., None] >> shifts) & np.uint32(0xFF)).astype(np.int64)
    return np.where(u >= 128, u - 256, u).reshape(w.shape[:-1] + (cols,))


_ORIG_DEQ = O.dequantize


def _dequant_group_of_int4_width(q, s, b, group, bits=4):
    # the group index computed as if 8 codes per word (columns of the int4 layout)
    if bits == 8:
        cols = q.shape[-1] * 4
        codes = O.unpack_int8(q, cols).astype(np.float64)
        gi = (np.arange(cols) // 2) // group
        return O.bf16_to_f64(s)[..., gi] * codes + O.bf16_to_f64(b)[..., gi]
    return _ORIG_DEQ(q, s, b, group, bits)


MUTATIONS = {
    "high_byte_first": ("unpack_int8", _unpack8_high_first),
    "seven_bit_mask": ("unpack_int8", _unpack8_seven_bits),
    "signed_codes": ("unpack_int8", _unpack8_signed),
    "group_index_halved": ("dequantize", _dequant_group_of_int4_width),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_int8_mutation_is_caught(name, monkeypatch, root):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = 0
    for pin in _pins(root):
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed, f"mutation {name} passed every int8 pin"
