"""A second, deliberately naive restatement of the MoE block in pure Python.

Used only to pin the oracle on tiny shapes.  It shares nothing with the
oracle: bf16 values are decoded with ``struct``, int4 codes with hexadecimal
digit strings, every logit is computed exactly with ``fractions.Fraction``
(no error bounds, no candidate pruning), and every product and sum is an
explicit Python loop.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def bf16(bits: int) -> float:
    return struct.unpack(">f", struct.pack(">I", (int(bits) & 0xFFFF) << 16))[0]


def f32(v) -> float:
    return struct.unpack(">f", struct.pack(">f", float(v)))[0]


def codes_of_word(word: int) -> list:
    # hex digits printed most-significant first; reversed -> bits 0..3 first
    return [int(c, 16) for c in format(int(word), "08x")[::-1]]


def codes_of_word8(word: int) -> list:
    # two hex digits per byte, most-significant byte first; reversed -> byte 0 first
    h = format(int(word), "08x")
    return [int(h[i:i + 2], 16) for i in (6, 4, 2, 0)]


def dequant_row(qrow, srow, brow, group: int, bits: int = 4) -> list:
    codes = []
    for w in qrow:
        codes.extend(codes_of_word(w) if bits == 4 else codes_of_word8(w))
    return [bf16(srow[c // group]) * codes[c] + bf16(brow[c // group]) for c in range(len(codes))]


def matvec(rows, vec) -> list:
    out = []
    for r in rows:
        acc = 0.0
        for a, b in zip(r, vec):
            acc += a * b
        out.append(acc)
    return out


def mlp(ex: dict, i: int, group: int, x: list, bits: int = 4) -> list:
    n_in = len(ex["gate_q"][i])
    gate = [dequant_row(ex["gate_q"][i][r], ex["gate_s"][i][r], ex["gate_b"][i][r], group, bits)
            for r in range(n_in)]
    up = [dequant_row(ex["up_q"][i][r], ex["up_s"][i][r], ex["up_b"][i][r], group, bits)
          for r in range(n_in)]
    down = [dequant_row(ex["down_q"][i][r], ex["down_s"][i][r], ex["down_b"][i][r], group, bits)
            for r in range(len(ex["down_q"][i]))]
    a = matvec(gate, x)
    u = matvec(up, x)
    h = [a[i_] / (1.0 + math.exp(-a[i_])) * u[i_] for i_ in range(len(a))]
    return matvec(down, h)


def block(x_bits, W: dict, k: int, group: int) -> dict:
    """y, topk_idx, topk_w, gate, perm, offsets for all tokens (lists)."""
    T = len(x_bits)
    E = len(W["router_w"])
    rb = W.get("router_bias")
    bits = W.get("bits", 4)
    ys, idxs, wss, gates = [], [], [], []
    for t in range(T):
        x = [bf16(v) for v in x_bits[t]]
        exact = []
        for e in range(E):
            acc = Fraction(0)
            for xv, wb in zip(x, W["router_w"][e]):
                acc += Fraction(xv) * Fraction(bf16(wb))
            if rb is not None:
                acc += Fraction(f32(rb[e]))
            exact.append(acc)
        order = sorted(range(E), key=lambda e: (-exact[e], e))
        sel = order[:k]
        fl = [float(v) for v in exact]
        m = max(fl)
        z = sum(math.exp(v - m) for v in fl)
        p = [math.exp(v - m) / z for v in fl]
        den = sum(p[e] for e in sel)
        w = [p[e] / den for e in sel]
        g = 1.0 / (1.0 + math.exp(-sum(a * bf16(b) for a, b in zip(x, W["shared_gate_w"]))))
        y = [0.0] * len(x)
        for j, e in enumerate(sel):
            o = mlp(W["experts"], e, group, x, bits)
            y = [y[h] + w[j] * o[h] for h in range(len(x))]
        s = mlp(W["shared"], 0, group, x, bits)
        y = [y[h] + g * s[h] for h in range(len(x))]
        ys.append(y)
        idxs.append(sel)
        wss.append(w)
        gates.append(g)
    flat = [e for row in idxs for e in row]
    perm = sorted(range(len(flat)), key=lambda p: (flat[p], p))
    offsets = [sum(1 for e in flat if e < b) for b in range(E + 1)]
    return {"y": ys, "topk_idx": idxs, "topk_w": wss, "gate": gates, "perm": perm,
            "offsets": offsets}


def bf16_round(v: float) -> int:
    """bf16 bits of float v, nearest with ties to even, from the float64 bit
    fields (integer arithmetic only)."""
    u = struct.unpack(">Q", struct.pack(">d", float(v)))[0]
    sign, exp, frac = u >> 63, (u >> 52) & 0x7FF, u & ((1 << 52) - 1)
    if exp == 0 and frac == 0:
        return sign << 15
    mant = (1 << 52) | frac            # 53 significant bits, value mant * 2^(exp - 1075)
    keep, drop = mant >> 45, mant & ((1 << 45) - 1)  # 8 bits kept
    half = 1 << 44
    if drop > half or (drop == half and keep & 1):
        keep += 1
    if keep == 1 << 8:                 # carried into a new binade
        keep >>= 1
        exp += 1
    e32 = exp - 1023 + 127             # float32 exponent field
    assert 0 < e32 < 255, v
    return (sign << 15) | (e32 << 7) | (keep & 0x7F)


def rms_norm(x_bits, g_bits, eps: float) -> list:
    x = [bf16(b) for b in x_bits]
    g = [1.0] * len(x) if g_bits is None else [bf16(b) for b in g_bits]
    ms = math.fsum(v * v for v in x) / len(x)
    d = math.sqrt(ms + eps)
    return [bf16_round(x[h] / d * g[h]) for h in range(len(x))]


def stack(x_bits, Ws: list, norm_ws, k: int, group: int, eps: float) -> dict:
    """One token through the blocks: n = rms_norm(x), x <- bf16(x + bf16(y))."""
    x = [int(b) for b in x_bits]
    out = {"x": [x], "xn": [], "y": [], "topk_idx": []}
    for l, W in enumerate(Ws):
        n = rms_norm(x, None if norm_ws is None else norm_ws[l], eps)
        r = block([n], W, k, group)
        y = r["y"][0]
        x = [bf16_round(bf16(x[h]) + bf16(bf16_round(y[h]))) for h in range(len(x))]
        out["xn"].append(n)
        out["y"].append(y)
        out["topk_idx"].append(r["topk_idx"][0])
        out["x"].append(x)
    return out
