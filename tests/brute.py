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


def dequant_row(qrow, srow, brow, group: int) -> list:
    codes = []
    for w in qrow:
        codes.extend(codes_of_word(w))
    return [bf16(srow[c // group]) * codes[c] + bf16(brow[c // group]) for c in range(len(codes))]


def matvec(rows, vec) -> list:
    out = []
    for r in rows:
        acc = 0.0
        for a, b in zip(r, vec):
            acc += a * b
        out.append(acc)
    return out


def mlp(ex: dict, i: int, group: int, x: list) -> list:
    n_in = len(ex["gate_q"][i])
    gate = [dequant_row(ex["gate_q"][i][r], ex["gate_s"][i][r], ex["gate_b"][i][r], group)
            for r in range(n_in)]
    up = [dequant_row(ex["up_q"][i][r], ex["up_s"][i][r], ex["up_b"][i][r], group)
          for r in range(n_in)]
    down = [dequant_row(ex["down_q"][i][r], ex["down_s"][i][r], ex["down_b"][i][r], group)
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
            o = mlp(W["experts"], e, group, x)
            y = [y[h] + w[j] * o[h] for h in range(len(x))]
        s = mlp(W["shared"], 0, group, x)
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
