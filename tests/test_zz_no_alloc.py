"""The allocation-free routing entry point against the regular one (GPU).

moe_route_static serves callers that cannot allocate device memory: it
keeps its intermediates in a library-owned static device array instead of a
workspace from cudaMalloc.  Its results must equal those of moe_forward, the
allocating entry point, on consecutive calls that reuse the shared array.
This file is collected last so that a failure here never hides another test.
"""
import numpy as np
import pytest

import int4_routed_expert_decode_gb300 as moe
import synth
from oracle import moe_oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def _dev(a, torch):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


@pytest.mark.parametrize("wid,T", [(0, 4), (3, 64)])
def test_static_routing_matches_moe_forward_on_two_calls(wid, T):
    import torch
    from int4_routed_expert_decode_gb300 import build
    build.build()
    wl = synth.WORKLOADS[wid]
    W = synth.layer_weights(0, wl.wid, 0, wl.shape, zipf_s=wl.zipf_s)
    layer = U.layer(wl.shape, W, max_T=T)
    rw = _dev(W["router_w"], torch)
    rb = _dev(W["router_bias"], torch)
    sg = _dev(W["shared_gate_w"], torch)
    for step in range(2):  # two calls in a row on the same static scratch
        x_np = synth.tokens(0, wl.wid, 0, 10 + step, T, wl.H)
        x = torch.from_numpy(x_np.view(np.int16)).cuda().view(torch.bfloat16)
        _, idx_ref, w_ref = layer.forward(x)
        idx = torch.full((T, wl.k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, wl.k), -1.0, dtype=torch.float32, device="cuda")
        g = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
        moe.moe_route_static(x, T, rw, rb, sg, wl.E, wl.k, wl.H, idx, w, g)
        torch.cuda.synchronize()
        assert layer.status() == moe.MOE_OK
        assert torch.equal(idx, idx_ref), f"call {step}: topk_idx differs from moe_forward"
        assert torch.max(torch.abs(w - w_ref)).item() <= U.W_ABS, f"call {step}: topk_w"
        # and directly against the CPU oracle's routing of the same tokens
        o_idx, o_w, o_gate, _ = O.route(x_np, W, wl.k)
        assert np.array_equal(idx.cpu().numpy(), o_idx), f"call {step}: topk_idx vs oracle"
        assert np.max(np.abs(w.cpu().numpy() - o_w)) <= U.W_ABS, f"call {step}: topk_w vs oracle"
        assert np.max(np.abs(g.cpu().numpy() - o_gate)) <= 1e-5, f"call {step}: shared gate"
    layer.close()


def test_static_routing_rejects_sizes_beyond_its_scratch():
    import torch
    from int4_routed_expert_decode_gb300 import build
    build.build()
    E, k, H = 512, 10, 2048
    x = torch.zeros((300, H), dtype=torch.bfloat16, device="cuda")
    rw = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    sg = torch.zeros((H,), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((300, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((300, k), dtype=torch.float32, device="cuda")
    g = torch.zeros((300,), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as e:  # 300 * 512 logits > 131072
        moe.moe_route_static(x, 300, rw, None, sg, E, k, H, idx, w, g)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    assert "static scratch limit" in moe.moe_last_error(None)
