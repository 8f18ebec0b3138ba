"""ctypes shim of the C++ CPU oracle (moe_oracle.cpp) -- TEST INFRASTRUCTURE ONLY.

``moe_block`` and ``moe_stack`` take and return the same things as the
functions of the same names in ``moe_oracle.py`` (the numpy restatement);
``threads`` sets the OpenMP thread count (0: the default).  The library is
compiled here with gcc on first use (``build()``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = SRC, out: str = LIB, force: bool = False) -> str:
    """Compile ``src`` into the shared library ``out`` (if stale) and return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.run(["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp],
                       check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """The compiled oracle (built on first use); ``path`` loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(L):
    P, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    L.oracle_bf16_round.argtypes = [P, ctypes.c_int64, P]
    L.oracle_bf16_round.restype = None
    L.oracle_moe_block.argtypes = [i32] * 7 + [P] * 10 + [P, i32, i32] + [P] * 7
    L.oracle_moe_block.restype = i32
    L.oracle_moe_stack.argtypes = [i32] * 7 + [P] * 5 + [f64] + [P] * 7 + [i32] + [P] * 5
    L.oracle_moe_stack.restype = i32
    return L


def _p(a) -> int | None:
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class _Weights:
    """Contiguous arrays of one layer's weights and the pointer tables to them."""

    def __init__(self, W: dict):
        self.rw = _c(W["router_w"], np.uint16)
        self.rb = _c(W.get("router_bias"), np.float32)
        self.gv = _c(W["shared_gate_w"], np.uint16)
        self.keep = []

        def table(part, kind, dtype):
            arrs = [_c(W[part][f"{m}_{kind}"], dtype) for m in ("gate", "up", "down")]
            self.keep.extend(arrs)
            return [a.ctypes.data for a in arrs]

        self.sq, self.ss, self.sb = (table("shared", "q", np.uint32), table("shared", "s", np.uint16),
                                     table("shared", "b", np.uint16))
        self.eq, self.es, self.eb = (table("experts", "q", np.uint32),
                                     table("experts", "s", np.uint16),
                                     table("experts", "b", np.uint16))
        self.E = self.rw.shape[0]
        self.Is = W["shared"]["gate_q"].shape[-2]
        self.I = W["experts"]["gate_q"].shape[-2]


def _ptrs(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def bf16_round(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    load().oracle_bf16_round(_p(v), v.size, _p(out))
    return out


def moe_block(x_bits, W: dict, k: int, group: int, tokens=None, threads: int = 0,
              lib=None) -> dict:
    L = lib or load()
    x = _c(x_bits, np.uint16)
    T, H = x.shape
    w = _Weights(W)
    toks = list(range(T)) if tokens is None else [int(t) for t in tokens]
    rows = np.array(toks, np.int32)
    y = np.zeros((len(toks), H))
    idx = np.zeros((T, k), np.int32)
    wts = np.zeros((T, k))
    gate = np.zeros(T)
    logits = np.zeros((T, w.E))
    perm = np.zeros(T * k, np.int32)
    offs = np.zeros(w.E + 1, np.int32)
    L.oracle_moe_block(T, H, w.E, k, w.I, w.Is, group, _p(x), _p(w.rw), _p(w.rb), _p(w.gv),
                       _ptrs(w.sq), _ptrs(w.ss), _ptrs(w.sb), _ptrs(w.eq), _ptrs(w.es),
                       _ptrs(w.eb), _p(rows), len(toks), threads, _p(y), _p(idx), _p(wts),
                       _p(gate), _p(logits), _p(perm), _p(offs))
    return {"y": y, "topk_idx": idx, "topk_w": wts, "shared_gate": gate, "perm": perm,
            "offsets": offs, "logits": logits, "tokens": toks}


def moe_stack(x_bits, Ws: list, norm_ws, k: int, group: int, eps: float, xn_given=None,
              threads: int = 0, lib=None) -> dict:
    L = lib or load()
    x = _c(np.asarray(x_bits).reshape(-1), np.uint16)
    H = x.shape[0]
    n = len(Ws)
    ws = [_Weights(W) for W in Ws]
    norms = [None if norm_ws is None or norm_ws[l] is None else _c(norm_ws[l], np.uint16)
             for l in range(n)]
    flat = lambda attr: _ptrs([p for w in ws for p in getattr(w, attr)])
    xs = np.zeros((n + 1, H), np.uint16)
    xn = np.zeros((n, H), np.uint16)
    y = np.zeros((n, H))
    idx = np.zeros((n, k), np.int32)
    wts = np.zeros((n, k))
    given = None if xn_given is None else _c(xn_given, np.uint16)
    L.oracle_moe_stack(n, H, ws[0].E, k, ws[0].I, ws[0].Is, group, _p(x),
                       _ptrs([_p(w.rw) for w in ws]), _ptrs([_p(w.rb) for w in ws]),
                       _ptrs([_p(w.gv) for w in ws]), _ptrs([_p(g) for g in norms]), eps,
                       flat("sq"), flat("ss"), flat("sb"), flat("eq"), flat("es"), flat("eb"),
                       _p(given), threads, _p(xs), _p(xn), _p(y), _p(idx), _p(wts))
    return {"x": xs, "xn": xn, "y": y, "topk_idx": idx, "topk_w": wts}
