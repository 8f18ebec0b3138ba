"""Python binding of the int4 routed-expert MoE block library (GB300, sm_103a).

A thin ``ctypes`` layer over ``libmoe_gb300.so`` (C ABI in ``include/moe.h``):
the functions below carry the C names and only marshal arguments; every step
of the block runs in the library's CUDA kernels.  PyTorch is used by callers
for device memory and streams only.  There is no fallback: if the shared
library is missing the first call raises ``MoEError``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_CUDA = -2
MOE_ERR_OOM = -3
MOE_ERR_NOT_LOADED = -4
MOE_ERR_NOT_RESERVED = -5
MOE_ERR_SLOT = -6
MOE_ERR_TIMEOUT = -7
MOE_ERR_UNSUPPORTED = -8

MOE_PATH_AUTO, MOE_PATH_DECODE, MOE_PATH_GENERAL, MOE_PATH_PREFILL = 0, 1, 2, 3
MOE_TEST_WAIT_TIMEOUT = 1
(MOE_MARK_START, MOE_MARK_LOGITS, MOE_MARK_ROUTED, MOE_MARK_PERMUTED, MOE_MARK_GATEUP,
 MOE_MARK_DOWN, MOE_MARK_END, MOE_MARK_COUNT) = range(8)

# every symbol include/moe.h declares
EXPORTS = (
    "moe_create", "moe_load_weights", "moe_reserve", "moe_forward", "moe_get_status",
    "moe_read_expert", "moe_set_path", "moe_expert_blob_bytes", "moe_device_bytes",
    "moe_last_launch_count", "moe_last_error", "moe_status_string", "moe_destroy",
    "moe_route_static", "moe_set_test_flags", "moe_set_stage_events", "moe_stack_create",
    "moe_stack_forward", "moe_stack_get_status", "moe_stack_set_test_flags", "moe_stack_destroy",
    "moe_router_check_stats", "moe_pool_enable", "moe_pool_stats", "moe_pool_table",
    "moe_gdn_recurrence", "moe_create_quant",
)


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


class QMatrix(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("b", ctypes.c_void_p)]


class Weights(ctypes.Structure):
    _fields_ = [
        ("on_device", ctypes.c_int),
        ("router_w", ctypes.c_void_p),
        ("router_bias", ctypes.c_void_p),
        ("shared_gate_w", ctypes.c_void_p),
        ("shared_gate", QMatrix), ("shared_up", QMatrix), ("shared_down", QMatrix),
        ("gate", QMatrix), ("up", QMatrix), ("down", QMatrix),
    ]


_lib = None


def lib():
    """Load the shared library (raises MoEError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise MoEError(MOE_ERR_CUDA, f"CUDA library not built: {LIB_PATH} is missing "
                                     "(run int4_routed_expert_decode_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    L.moe_create.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
    L.moe_create_quant.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
    L.moe_create_quant.restype = i32
    L.moe_load_weights.argtypes = [vp, ctypes.POINTER(Weights), i32, vp]
    L.moe_reserve.argtypes = [vp, i32]
    L.moe_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
    L.moe_get_status.argtypes = [vp, vp]
    L.moe_read_expert.argtypes = [vp, i32] + [vp] * 9
    L.moe_set_path.argtypes = [vp, i32]
    L.moe_set_test_flags.argtypes = [vp, i32]
    L.moe_set_stage_events.argtypes = [vp, ctypes.POINTER(vp), i32]
    L.moe_expert_blob_bytes.argtypes = [vp]
    L.moe_expert_blob_bytes.restype = i64
    L.moe_device_bytes.argtypes = [vp]
    L.moe_device_bytes.restype = i64
    L.moe_last_launch_count.argtypes = [vp]
    L.moe_last_error.argtypes = [vp]
    L.moe_last_error.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [i32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_destroy.argtypes = [vp]
    L.moe_destroy.restype = None
    L.moe_route_static.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp]
    L.moe_route_static.restype = i32
    L.moe_stack_create.argtypes = [ctypes.POINTER(vp), i32, ctypes.POINTER(vp), ctypes.c_float,
                                   ctypes.POINTER(vp)]
    L.moe_stack_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_stack_get_status.argtypes = [vp, vp]
    L.moe_stack_set_test_flags.argtypes = [vp, i32]
    L.moe_router_check_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_int)]
    L.moe_router_check_stats.restype = i32
    L.moe_pool_enable.argtypes = [vp, i32]
    L.moe_pool_enable.restype = i32
    L.moe_pool_stats.argtypes = [vp, vp]
    L.moe_pool_stats.restype = i32
    L.moe_pool_table.argtypes = [vp, vp]
    L.moe_pool_table.restype = i32
    L.moe_stack_destroy.argtypes = [vp]
    L.moe_gdn_recurrence.argtypes = [vp] * 7 + [i32] * 6 + [vp]
    L.moe_gdn_recurrence.restype = i32
    L.moe_stack_destroy.restype = None
    for name in ("moe_create", "moe_load_weights", "moe_reserve", "moe_forward", "moe_get_status",
                 "moe_read_expert", "moe_set_path", "moe_last_launch_count",
                 "moe_set_test_flags", "moe_set_stage_events", "moe_stack_create",
                 "moe_stack_forward", "moe_stack_get_status", "moe_stack_set_test_flags"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def _check(status: int, ctx=None) -> int:
    if status != MOE_OK:
        msg = lib().moe_last_error(ctx)
        raise MoEError(status, msg.decode() if msg else lib().moe_status_string(status).decode())
    return status


def _addr(a) -> int | None:
    """Address of a torch tensor, numpy array or int (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"], "arrays must be contiguous"
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        assert a.is_contiguous(), "tensors must be contiguous"
        return a.data_ptr()
    raise TypeError(f"cannot take the address of {type(a)}")


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- C-named calls
def moe_create(E, k, hidden, inter, shared_inter, group) -> int:
    out = ctypes.c_void_p()
    _check(lib().moe_create(E, k, hidden, inter, shared_inter, group, ctypes.byref(out)))
    return out.value


def moe_create_quant(E, k, hidden, inter, shared_inter, group, bits) -> int:
    out = ctypes.c_void_p()
    _check(lib().moe_create_quant(E, k, hidden, inter, shared_inter, group, bits,
                                  ctypes.byref(out)))
    return out.value


def make_weights(W: dict, on_device: bool) -> tuple[Weights, list]:
    """moe_weights from a dict of canonical arrays (numpy for host, torch for device).

    Keys: router_w, router_bias (or None), shared_gate_w, shared{gate,up,down}_{q,s,b},
    experts{...}.  Returns the struct and the list of arrays it points into (keep
    it alive until moe_load_weights returns).
    """
    keep = []

    def a(v):
        if v is None:
            return None
        if isinstance(v, np.ndarray):
            v = np.ascontiguousarray(v)
        elif hasattr(v, "contiguous"):
            v = v.contiguous()
        keep.append(v)
        return _addr(v)

    def qm(d, name):
        return QMatrix(a(d[name + "_q"]), a(d[name + "_s"]), a(d[name + "_b"]))

    w = Weights(1 if on_device else 0, a(W["router_w"]), a(W.get("router_bias")),
                a(W["shared_gate_w"]), qm(W["shared"], "gate"), qm(W["shared"], "up"),
                qm(W["shared"], "down"), qm(W["experts"], "gate"), qm(W["experts"], "up"),
                qm(W["experts"], "down"))
    return w, keep


def moe_load_weights(ctx: int, W: dict, n_slots: int, on_device: bool = False, stream=None):
    w, keep = make_weights(W, on_device)
    _check(lib().moe_load_weights(ctx, ctypes.byref(w), n_slots, _stream(stream)), ctx)
    del keep


def moe_reserve(ctx: int, max_T: int):
    _check(lib().moe_reserve(ctx, max_T), ctx)


def moe_forward(ctx: int, x, T: int, expert_slot_table, y, topk_idx, topk_w, perm=None,
                offsets=None, stream=None):
    _check(lib().moe_forward(ctx, _addr(x), T, _addr(expert_slot_table), _addr(y),
                             _addr(topk_idx), _addr(topk_w), _addr(perm), _addr(offsets),
                             _stream(stream)), ctx)


def moe_get_status(ctx: int, stream=None) -> int:
    """Synchronise and return the sticky device status (does not raise)."""
    return lib().moe_get_status(ctx, _stream(stream))


def moe_read_expert(ctx: int, slot: int, H: int, I: int, G: int, bits: int = 4) -> dict:
    c = 32 // bits  # codes per packed word
    out = {
        "gate_q": np.empty((I, H // c), np.uint32), "gate_s": np.empty((I, H // G), np.uint16),
        "gate_b": np.empty((I, H // G), np.uint16), "up_q": np.empty((I, H // c), np.uint32),
        "up_s": np.empty((I, H // G), np.uint16), "up_b": np.empty((I, H // G), np.uint16),
        "down_q": np.empty((H, I // c), np.uint32), "down_s": np.empty((H, I // G), np.uint16),
        "down_b": np.empty((H, I // G), np.uint16),
    }
    order = ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s", "down_b")
    _check(lib().moe_read_expert(ctx, slot, *[_addr(out[k]) for k in order]), ctx)
    return out


def moe_set_path(ctx: int, path: int):
    _check(lib().moe_set_path(ctx, path), ctx)


def moe_set_test_flags(ctx: int, flags: int):
    _check(lib().moe_set_test_flags(ctx, flags), ctx)


def moe_set_stage_events(ctx: int, events):
    """Borrow cudaEvent_t handles (ints, or torch.cuda.Event objects that have
    been recorded once, so that they exist) for the stage marks; [] turns
    the marks off."""
    hs = [e if isinstance(e, int) else int(e.cuda_event) for e in events]
    arr = (ctypes.c_void_p * max(1, len(hs)))(*hs)
    _check(lib().moe_set_stage_events(ctx, arr if hs else None, len(hs)), ctx)


def moe_expert_blob_bytes(ctx: int) -> int:
    return int(lib().moe_expert_blob_bytes(ctx))


def moe_device_bytes(ctx: int) -> int:
    return int(lib().moe_device_bytes(ctx))


def moe_last_launch_count(ctx: int) -> int:
    return int(lib().moe_last_launch_count(ctx))


def moe_last_error(ctx: int | None) -> str:
    m = lib().moe_last_error(ctx)
    return m.decode() if m else ""


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_destroy(ctx: int):
    lib().moe_destroy(ctx)


def moe_route_static(x, T: int, router_w, router_bias, shared_gate_w, E: int, k: int,
                     hidden: int, topk_idx, topk_w, shared_gate, stream=None):
    """Routing with no allocation (library-owned static scratch); see include/moe.h."""
    _check(lib().moe_route_static(_addr(x), T, _addr(router_w), _addr(router_bias),
                                  _addr(shared_gate_w), E, k, hidden, _addr(topk_idx),
                                  _addr(topk_w), _addr(shared_gate), _stream(stream)))


def moe_gdn_recurrence(q, k, v, alpha, beta, state, out, B: int, T: int, Hk: int, Hv: int,
                       dk: int, dv: int, stream=None):
    """Gated DeltaNet recurrence over B sequences of T tokens, state updated in
    place (device pointers or tensors); see include/moe.h."""
    _check(lib().moe_gdn_recurrence(_addr(q), _addr(k), _addr(v), _addr(alpha), _addr(beta),
                                    _addr(state), _addr(out), B, T, Hk, Hv, dk, dv,
                                    _stream(stream)))


def moe_pool_enable(ctx: int, slots: int):
    _check(lib().moe_pool_enable(ctx, slots), ctx)


def moe_pool_stats(ctx: int) -> dict:
    out = np.zeros(5, np.int64)
    _check(lib().moe_pool_stats(ctx, out.ctypes.data), ctx)
    return {"calls": int(out[0]), "hits": int(out[1]), "misses": int(out[2]),
            "evictions": int(out[3]), "overflows": int(out[4])}


def moe_pool_table(ctx: int, E: int) -> np.ndarray:
    out = np.zeros(E, np.int32)
    _check(lib().moe_pool_table(ctx, out.ctypes.data), ctx)
    return out


def moe_router_check_stats(ctx: int) -> tuple[float, int]:
    """(largest measured tensor-core router error / (|x| max|Wr|), fallback tokens)
    since the last read; resets both (see include/moe.h)."""
    r, n = ctypes.c_float(), ctypes.c_int()
    _check(lib().moe_router_check_stats(ctx, ctypes.byref(r), ctypes.byref(n)), ctx)
    return r.value, n.value


def moe_stack_create(layer_ctxs, norm_w=None, eps: float = 1e-6) -> int:
    """A stack over contexts `layer_ctxs` (see include/moe.h); norm_w: None or a
    list of device bf16 [H] tensors / addresses (None entries: all ones)."""
    n = len(layer_ctxs)
    ctxs = (ctypes.c_void_p * n)(*layer_ctxs)
    norms = None
    if norm_w is not None:
        norms = (ctypes.c_void_p * n)(*[_addr(w) for w in norm_w])
    out = ctypes.c_void_p()
    _check(lib().moe_stack_create(ctxs, n, norms, ctypes.c_float(eps), ctypes.byref(out)))
    return out.value


def moe_stack_forward(stack: int, x, expert_slot_tables, x_out, y, xn, topk_idx, topk_w,
                      stream=None):
    _check(lib().moe_stack_forward(stack, _addr(x), _addr(expert_slot_tables), _addr(x_out),
                                   _addr(y), _addr(xn), _addr(topk_idx), _addr(topk_w),
                                   _stream(stream)))


def moe_stack_get_status(stack: int, stream=None) -> int:
    """Synchronise and return the stack's sticky device status (does not raise)."""
    return lib().moe_stack_get_status(stack, _stream(stream))


def moe_stack_set_test_flags(stack: int, flags: int):
    _check(lib().moe_stack_set_test_flags(stack, flags))


def moe_stack_destroy(stack: int):
    lib().moe_stack_destroy(stack)


# ----------------------------------------------------------------- convenience
class MoEStack:
    """L loaded MoELayers of one shape chained for one token in one launch.

    ``forward(x)`` takes a CUDA bf16 tensor [H] and returns (x_out [H],
    y [L, H], xn [L, H], topk_idx [L, k], topk_w [L, k]).
    """

    def __init__(self, layers, norm_w=None, eps: float = 1e-6):
        self.layers = list(layers)  # kept alive: the stack borrows their weights
        self.L = len(self.layers)
        l0 = self.layers[0]
        self.H, self.k, self.E = l0.H, l0.k, l0.E
        self.norm_w = norm_w
        self.stack = moe_stack_create([l.ctx for l in self.layers], norm_w, eps)

    def forward(self, x, tables=None, x_out=None, y=None, xn=None, topk_idx=None, topk_w=None,
                stream=None):
        import torch
        dev = x.device
        if x_out is None:
            x_out = torch.empty((self.H,), dtype=torch.bfloat16, device=dev)
        if y is None:
            y = torch.empty((self.L, self.H), dtype=torch.bfloat16, device=dev)
        if xn is None:
            xn = torch.empty((self.L, self.H), dtype=torch.bfloat16, device=dev)
        if topk_idx is None:
            topk_idx = torch.empty((self.L, self.k), dtype=torch.int32, device=dev)
        if topk_w is None:
            topk_w = torch.empty((self.L, self.k), dtype=torch.float32, device=dev)
        moe_stack_forward(self.stack, x, tables, x_out, y, xn, topk_idx, topk_w, stream)
        return x_out, y, xn, topk_idx, topk_w

    def status(self, stream=None) -> int:
        return moe_stack_get_status(self.stack, stream)

    def close(self):
        if self.stack:
            moe_stack_destroy(self.stack)
            self.stack = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoELayer:
    """One MoE layer: a context with its weights and workspace.

    ``forward(x)`` takes a CUDA bf16 tensor [T, H] and returns
    (y bf16 [T, H], topk_idx int32 [T, k], topk_w fp32 [T, k]); ``perm`` and
    ``offsets`` may be passed to receive the permutation as well.
    """

    def __init__(self, E, k, H, I, Is, G, weights: dict | None = None, n_slots=None,
                 max_T=1, on_device=False, bits=4):
        self.E, self.k, self.H, self.I, self.Is, self.G = E, k, H, I, Is, G
        self.bits = bits
        self.ctx = moe_create_quant(E, k, H, I, Is, G, bits)
        if weights is not None:
            self.load(weights, n_slots or E, on_device)
        moe_reserve(self.ctx, max_T)

    def load(self, weights: dict, n_slots: int, on_device=False):
        moe_load_weights(self.ctx, weights, n_slots, on_device)

    def forward(self, x, table=None, y=None, topk_idx=None, topk_w=None, perm=None,
                offsets=None, stream=None):
        import torch
        T = x.shape[0]
        dev = x.device
        if y is None:
            y = torch.empty((T, self.H), dtype=torch.bfloat16, device=dev)
        if topk_idx is None:
            topk_idx = torch.empty((T, self.k), dtype=torch.int32, device=dev)
        if topk_w is None:
            topk_w = torch.empty((T, self.k), dtype=torch.float32, device=dev)
        moe_forward(self.ctx, x, T, table, y, topk_idx, topk_w, perm, offsets, stream)
        return y, topk_idx, topk_w

    def status(self, stream=None) -> int:
        return moe_get_status(self.ctx, stream)

    def close(self):
        if self.ctx:
            moe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
