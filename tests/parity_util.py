"""Helpers of the GPU parity tests: load synthetic weights into the library,
run it, and compare with the CPU oracle at the block's tolerances.

Tolerances (bf16 outputs, fp32 accumulation):
  * topk_idx, perm, offsets: bit-exact;
  * y: max|y - y_ref| <= 2e-2 * max|y_ref| and sum|y - y_ref| / sum|y_ref| <= 5e-3;
  * topk_w: |w - w_ref| <= 1e-5 (fp32 weights summing to one).
"""
from __future__ import annotations

import numpy as np

import int4_routed_expert_decode_gb300 as moe

Y_MAX_REL = 2e-2
Y_MEAN_REL = 5e-3
W_ABS = 1e-5


def to_f64_bf16(t) -> np.ndarray:
    """A torch bf16 tensor -> float64 numpy (exact)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def layer(shape, W, max_T, n_slots=None, device_weights=False):
    L = moe.MoELayer(shape.E, shape.k, shape.H, shape.I, shape.Is, shape.G, max_T=max_T,
                     bits=int(W.get("bits", 4)))
    if device_weights:
        import torch
        W = to_device(W)
    L.load(W, n_slots or shape.E, on_device=device_weights)
    return L


def to_device(W):
    import torch

    def t(a):
        if a is None:
            return None
        if a.dtype == np.uint32:
            return torch.from_numpy(a.view(np.int32)).cuda()
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).cuda()
        return torch.from_numpy(a).cuda()

    return {"router_w": t(W["router_w"]), "router_bias": t(W.get("router_bias")),
            "shared_gate_w": t(W["shared_gate_w"]),
            "shared": {k: t(v) for k, v in W["shared"].items()},
            "experts": {k: t(v) for k, v in W["experts"].items()}}


def run(L, x_np, table=None, want_perm=True):
    """Run one forward on the GPU; returns numpy outputs."""
    import torch
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).cuda().view(torch.bfloat16)
    perm = torch.full((T * L.k,), -1, dtype=torch.int32, device="cuda") if want_perm else None
    offs = torch.full((L.E + 1,), -1, dtype=torch.int32, device="cuda") if want_perm else None
    tab = None if table is None else torch.as_tensor(table, dtype=torch.int32).cuda()
    y, idx, w = L.forward(x, table=tab, perm=perm, offsets=offs)
    status = L.status()
    out = {"y": to_f64_bf16(y), "topk_idx": idx.cpu().numpy(), "topk_w": w.cpu().numpy(),
           "status": status, "y_bits": y.view(torch.int16).cpu().numpy()}
    if want_perm:
        out["perm"] = perm.cpu().numpy()
        out["offsets"] = offs.cpu().numpy()
    return out


def y_errors(y, y_ref):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    d = np.abs(y - y_ref)
    return float(d.max() / np.abs(y_ref).max()), float(d.sum() / np.abs(y_ref).sum())


def assert_y_close(y, y_ref, what=""):
    mx, mean = y_errors(y, y_ref)
    assert mx <= Y_MAX_REL, f"{what} max rel err {mx:.3e} > {Y_MAX_REL}"
    assert mean <= Y_MEAN_REL, f"{what} mean rel err {mean:.3e} > {Y_MEAN_REL}"
    return mx, mean


def assert_parity(out, ref, rows=None, check_perm=True, what=""):
    assert out["status"] == moe.MOE_OK, moe.moe_status_string(out["status"])
    assert np.array_equal(out["topk_idx"], ref["topk_idx"]), f"{what} topk_idx differs"
    assert np.max(np.abs(out["topk_w"] - ref["topk_w"])) <= W_ABS, f"{what} topk_w"
    if check_perm:
        assert np.array_equal(out["perm"], ref["perm"]), f"{what} perm differs"
        assert np.array_equal(out["offsets"], ref["offsets"]), f"{what} offsets differ"
    y = out["y"] if rows is None else out["y"][rows]
    return assert_y_close(y, ref["y"], what)
