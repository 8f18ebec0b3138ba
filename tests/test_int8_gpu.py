"""GPU parity of int8 experts (moe_create_quant with bits = 8) against the
oracle: the general path for every T, the slot pool, the expert read-back,
and the int4-only paths refusing the context."""
import numpy as np
import pytest

import int4_routed_expert_decode_gb300 as moe
import synth
from oracle import moe_oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_decode_gb300 import build
    build.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.init()


@pytest.mark.parametrize("wid,T", [(0, 1), (0, 3), (0, 4), (0, 33), (1, 1), (1, 8), (2, 1)])
def test_int8_block_matches_oracle(wid, T):
    wl = synth.WORKLOADS[wid]
    W = synth.layer_weights_int8(0, wl.wid, 90, wl.shape, zipf_s=wl.zipf_s)
    L = U.layer(wl.shape, W, max_T=T)
    x = synth.tokens(0, wl.wid, 90, 0, T, wl.H)
    out = U.run(L, x)
    rows = list(range(min(T, 6)))
    ref = O.moe_block(x, W, wl.k, wl.G, tokens=rows)
    U.assert_parity(out, ref, rows=rows, what=f"int8 wl{wid} T={T}")
    L.close()


def test_int8_group_128_and_deterministic():
    shape = synth.Shape(E=32, k=4, H=1024, I=256, Is=384, G=128)
    W = synth.layer_weights_int8(0, 0, 91, shape)
    L = U.layer(shape, W, max_T=5)
    x = synth.tokens(0, 0, 91, 0, 5, shape.H)
    a, b = U.run(L, x), U.run(L, x)
    assert np.array_equal(a["y_bits"], b["y_bits"])
    U.assert_parity(a, O.moe_block(x, W, shape.k, shape.G), what="int8 G=128")
    L.close()


def test_int8_read_back_is_the_canonical_weights():
    wl = synth.WORKLOADS[0]
    W = synth.layer_weights_int8(0, wl.wid, 92, wl.shape)
    L = U.layer(wl.shape, W, max_T=1)
    for slot, src, i in ((3, W["experts"], 3), (-1, W["shared"], 0)):
        got = moe.moe_read_expert(L.ctx, slot, wl.H, wl.Is if slot < 0 else wl.I, wl.G, bits=8)
        for key in ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s",
                    "down_b"):
            assert np.array_equal(got[key], src[key][i]), (slot, key)
    L.close()


def test_int8_pool_matches_oracle_across_evictions():
    wl = synth.WORKLOADS[0]
    W = synth.layer_weights_int8(0, wl.wid, 93, wl.shape)
    L = U.layer(wl.shape, W, max_T=2)
    moe.moe_pool_enable(L.ctx, 6)
    for step in range(6):
        x = synth.tokens(0, wl.wid, 93, step, 2, wl.H)
        U.assert_parity(U.run(L, x), O.moe_block(x, W, wl.k, wl.G), what=f"pool step {step}")
    st = moe.moe_pool_stats(L.ctx)
    assert st["misses"] > 0 and st["calls"] == 6
    L.close()


def test_int8_refuses_the_int4_only_paths():
    wl = synth.WORKLOADS[1]
    W = synth.layer_weights_int8(0, wl.wid, 94, wl.shape)
    L = U.layer(wl.shape, W, max_T=4)
    x = synth.tokens(0, wl.wid, 94, 0, 1, wl.H)
    for path in (moe.MOE_PATH_DECODE, moe.MOE_PATH_PREFILL):
        moe.moe_set_path(L.ctx, path)
        with pytest.raises(moe.MoEError) as e:
            U.run(L, x)
        assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    moe.moe_set_path(L.ctx, moe.MOE_PATH_AUTO)
    with pytest.raises(moe.MoEError) as e:
        moe.MoEStack([L], None, 1e-6)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    L.close()
