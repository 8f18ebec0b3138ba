"""Seeded synthetic inputs of the sparse int4 MoE block.

A module of its own: the CPU oracle and the CUDA library both consume the
arrays built here, and this module holds none of the block's arithmetic.  The
random numbers come from the counter-based SplitMix64 generator in
``synth.c`` (built on first use with gcc); the Zipf router prior is a plain
vector of log-weights.

Storage conventions (the MLX affine quantised layout):
  * bf16 tensors are ``numpy.uint16`` arrays holding the bf16 bit patterns;
  * packed int4 codes are ``numpy.uint32`` words, code ``8c+j`` of a row in
    bits ``4j..4j+3`` of word ``c`` (low nibble first);
  * a quantised matrix ``[rows, cols]`` is ``q [rows, cols/8]`` plus
    ``s, b [rows, cols/group]`` with ``w = s*q + b`` per group along ``cols``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile
from dataclasses import dataclass

import numpy as np

from .workloads import WORKLOADS, Workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (atomic replace)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_LIB_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
    lib.synth_draw.restype = u64
    lib.synth_draw.argtypes = [u64, u64]
    lib.synth_key.restype = u64
    lib.synth_key.argtypes = [u64, u64, u64, u64, u64]
    lib.synth_fill_u32.argtypes = [u64, i64, p]
    lib.synth_fill_normal_bf16.argtypes = [u64, i64, ctypes.c_double, ctypes.c_double, p]
    lib.synth_fill_scale_bias.argtypes = [u64, i64, p, p]
    lib.synth_fill_experts.argtypes = [u64, u64, u64, ctypes.c_int, i64, i64, i64, i64, i64,
                                       p, p, p, p, p, p, p, p, p]
    lib.synth_fill_router.argtypes = [u64, u64, u64, i64, i64, p, p]
    lib.synth_fill_tokens.argtypes = [u64, u64, u64, u64, i64, i64, p]
    for f in ("synth_fill_u32", "synth_fill_normal_bf16", "synth_fill_scale_bias",
              "synth_fill_experts", "synth_fill_router", "synth_fill_tokens"):
        getattr(lib, f).restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def draw(key: int, i: int) -> int:
    """Output ``i`` of the SplitMix64 sequence started at ``key``."""
    return int(_load().synth_draw(key, i))


def stream_key(seed: int, workload: int, layer: int, tensor: int, index: int) -> int:
    return int(_load().synth_key(seed, workload, layer, tensor, index))


def uniform_u32(key: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint32)
    _load().synth_fill_u32(key, n, _ptr(out))
    return out


def normal_bf16(key: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _load().synth_fill_normal_bf16(key, n, mean, std, _ptr(out))
    return out


def scale_bias(key: int, n: int):
    s = np.empty(n, np.uint16)
    b = np.empty(n, np.uint16)
    _load().synth_fill_scale_bias(key, n, _ptr(s), _ptr(b))
    return s, b


@dataclass(frozen=True)
class Shape:
    """Sizes of one MoE block: E experts, top-k, hidden H, expert inter I,
    shared-expert inter Is, quantisation group G."""
    E: int
    k: int
    H: int
    I: int
    Is: int
    G: int


def experts(seed: int, workload: int, layer: int, shape: Shape, e0: int = 0,
            n: int | None = None, shared: bool = False) -> dict:
    """Quantised expert tensors, canonical layout with a leading expert dim ``n``."""
    H, G = shape.H, shape.G
    I = shape.Is if shared else shape.I
    if n is None:
        n = 1 if shared else shape.E
    if shared:
        assert n == 1
    out = {
        "gate_q": np.empty((n, I, H // 8), np.uint32),
        "gate_s": np.empty((n, I, H // G), np.uint16),
        "gate_b": np.empty((n, I, H // G), np.uint16),
        "up_q": np.empty((n, I, H // 8), np.uint32),
        "up_s": np.empty((n, I, H // G), np.uint16),
        "up_b": np.empty((n, I, H // G), np.uint16),
        "down_q": np.empty((n, H, I // 8), np.uint32),
        "down_s": np.empty((n, H, I // G), np.uint16),
        "down_b": np.empty((n, H, I // G), np.uint16),
    }
    o = out
    _load().synth_fill_experts(seed, workload, layer, 1 if shared else 0, e0, n, H, I, G,
                               _ptr(o["gate_q"]), _ptr(o["gate_s"]), _ptr(o["gate_b"]),
                               _ptr(o["up_q"]), _ptr(o["up_s"]), _ptr(o["up_b"]),
                               _ptr(o["down_q"]), _ptr(o["down_s"]), _ptr(o["down_b"]))
    return out


def zipf_log_prior(E: int, s: float) -> np.ndarray:
    """Log of a Zipf(s) prior over experts, ranked by index: ``-s*ln(e+1)`` (float32)."""
    return np.array([-s * math.log(e + 1.0) for e in range(E)], dtype=np.float64).astype(np.float32)


def layer_weights(seed: int, workload: int, layer: int, shape: Shape,
                  zipf_s: float | None = None) -> dict:
    """All weights of one MoE layer in the canonical layout.

    Keys: ``router_w`` bf16 [E,H]; ``router_bias`` float32 [E] or None;
    ``shared_gate_w`` bf16 [H]; ``shared`` (dict, leading dim 1); ``experts``
    (dict, leading dim E).
    """
    rw = np.empty((shape.E, shape.H), np.uint16)
    sg = np.empty(shape.H, np.uint16)
    _load().synth_fill_router(seed, workload, layer, shape.E, shape.H, _ptr(rw), _ptr(sg))
    return {
        "router_w": rw,
        "router_bias": None if zipf_s is None else zipf_log_prior(shape.E, zipf_s),
        "shared_gate_w": sg,
        "shared": experts(seed, workload, layer, shape, shared=True),
        "experts": experts(seed, workload, layer, shape),
    }


def to_int8_experts(seed: int, workload: int, layer: int, ex: dict, shared: bool) -> dict:
    """int8 experts of the same sizes drawn from the int4 ones: codes uniform in
    0..255 (4 per word, fresh streams, tensor ids 37-39), scales s/16 (the int4
    scale with its bf16 exponent lowered by 4: weights of the same spread) and
    the int4 biases unchanged (= -128 times the new scale, so code 128 is 0)."""
    out = {}
    for i, name in enumerate(("gate", "up", "down")):
        q4 = ex[name + "_q"]
        n = q4.size * 2
        key = stream_key(seed, workload, layer, 37 + i, 1 if shared else 0)
        out[name + "_q"] = uniform_u32(key, n).reshape(q4.shape[:-1] + (q4.shape[-1] * 2,))
        out[name + "_s"] = (ex[name + "_s"].astype(np.int32) - (4 << 7)).astype(np.uint16)
        out[name + "_b"] = ex[name + "_b"].copy()
    return out


def layer_weights_int8(seed: int, workload: int, layer: int, shape: Shape,
                       zipf_s: float | None = None) -> dict:
    """As layer_weights, with int8 experts (``bits`` = 8)."""
    W = layer_weights(seed, workload, layer, shape, zipf_s=zipf_s)
    W["experts"] = to_int8_experts(seed, workload, layer, W["experts"], False)
    W["shared"] = to_int8_experts(seed, workload, layer, W["shared"], True)
    W["bits"] = 8
    return W


T_NORM_W = 30  # tensor id of the stacks' RMSNorm weights (ids below 30 are the C generator's)


def norm_weights(seed: int, workload: int, layer: int, H: int) -> np.ndarray:
    """RMSNorm weights of one layer of a stack, bf16 [H] ~ N(1, 0.1^2)."""
    return normal_bf16(stream_key(seed, workload, layer, T_NORM_W, 0), H, 1.0, 0.1)


def tokens(seed: int, workload: int, layer: int, step: int, T: int, H: int) -> np.ndarray:
    """Token activations bf16 [T, H] ~ N(0,1) for one (layer, step)."""
    x = np.empty((T, H), np.uint16)
    _load().synth_fill_tokens(seed, workload, layer, step, T, H, _ptr(x))
    return x


# Tensor ids of the Gated DeltaNet recurrence inputs.
T_GDN_Q, T_GDN_K, T_GDN_V, T_GDN_ALPHA, T_GDN_BETA, T_GDN_STATE = 31, 32, 33, 34, 35, 36


def uniform_f32(key: int, n: int, lo: float, hi: float) -> np.ndarray:
    """n float32 values uniform in [lo, hi): the top 24 bits of each draw."""
    u = (uniform_u32(key, n) >> np.uint32(8)).astype(np.float64) * (1.0 / (1 << 24))
    return (lo + (hi - lo) * u).astype(np.float32)


@dataclass(frozen=True)
class GdnShape:
    """Sizes of one Gated DeltaNet layer's recurrence: Hk key heads, Hv value
    heads (a multiple of Hk), key dim dk, value dim dv."""
    Hk: int = 16
    Hv: int = 32
    dk: int = 128
    dv: int = 128


def gdn_inputs(seed: int, layer: int, B: int, T: int, s: GdnShape, step: int = 0,
               alpha_lo: float = 0.80, state_std: float = 0.5):
    """Inputs of B independent sequences, T tokens each:
    q, k bf16 [B,T,Hk,dk] ~ N(0,1); v bf16 [B,T,Hv,dv] ~ N(0,1);
    alpha f32 [B,T,Hv] uniform in [alpha_lo, 1); beta f32 [B,T,Hv] uniform in [0, 1);
    state f32 [B,Hv,dv,dk] ~ N(0, state_std^2) (bf16 values widened)."""
    def key(t):
        return stream_key(seed, 9, layer, t, step)
    nq = B * T * s.Hk * s.dk
    q = normal_bf16(key(T_GDN_Q), nq).reshape(B, T, s.Hk, s.dk)
    k = normal_bf16(key(T_GDN_K), nq).reshape(B, T, s.Hk, s.dk)
    v = normal_bf16(key(T_GDN_V), B * T * s.Hv * s.dv).reshape(B, T, s.Hv, s.dv)
    alpha = uniform_f32(key(T_GDN_ALPHA), B * T * s.Hv, alpha_lo, 1.0).reshape(B, T, s.Hv)
    beta = uniform_f32(key(T_GDN_BETA), B * T * s.Hv, 0.0, 1.0).reshape(B, T, s.Hv)
    sb = normal_bf16(key(T_GDN_STATE), B * s.Hv * s.dv * s.dk, 0.0, state_std)
    state = (sb.astype(np.uint32) << 16).view(np.float32).reshape(B, s.Hv, s.dv, s.dk)
    return q, k, v, alpha, beta, state
