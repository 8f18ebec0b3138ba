"""GPU parity of the batched decode kernels (2 <= T <= 64 tokens: the used
experts' weights streamed once, their tokens in the MMA's N columns)."""
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


@pytest.mark.parametrize("wid,T", [(0, 2), (0, 4), (1, 5), (1, 33), (2, 17), (3, 64)])
def test_batched_decode_matches_oracle(wid, T):
    wl = synth.WORKLOADS[wid]
    W = synth.layer_weights(0, wl.wid, 80, wl.shape, zipf_s=wl.zipf_s)
    L = U.layer(wl.shape, W, max_T=T)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    x = synth.tokens(0, wl.wid, 80, 0, T, wl.H)
    out = U.run(L, x)
    assert moe.moe_last_launch_count(L.ctx) >= 4
    rows = list(range(min(T, 12)))
    ref = O.moe_block(x, W, wl.k, wl.G, tokens=rows)
    U.assert_parity(out, ref, rows=rows, what=f"batched wl{wid} T={T}")
    L.close()


def test_batched_decode_other_shapes():
    """Group 128 with hidden 1024, and inner sizes whose chunk counts are not
    powers of two (inter 192: unswizzled 96-byte down rows)."""
    for shape, T in ((synth.Shape(E=64, k=6, H=1024, I=256, Is=256, G=128), 9),
                     (synth.Shape(E=32, k=4, H=512, I=192, Is=192, G=64), 20)):
        W = synth.layer_weights(0, 0, 81, shape, zipf_s=0.5)
        L = U.layer(shape, W, max_T=T)
        moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
        x = synth.tokens(0, 0, 81, 0, T, shape.H)
        U.assert_parity(U.run(L, x), O.moe_block(x, W, shape.k, shape.G), what=f"{shape} T={T}")
        L.close()


def test_batched_decode_deterministic_and_equals_single_tokens():
    wl = synth.WORKLOADS[1]
    W = synth.layer_weights(0, wl.wid, 82, wl.shape)
    T = 6
    L = U.layer(wl.shape, W, max_T=T)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    x = synth.tokens(0, wl.wid, 82, 0, T, wl.H)
    a, b = U.run(L, x), U.run(L, x)
    assert np.array_equal(a["y_bits"], b["y_bits"])
    for t in range(T):
        one = U.run(L, x[t:t + 1])
        assert np.array_equal(one["topk_idx"][0], a["topk_idx"][t])
        U.assert_y_close(a["y"][t:t + 1], one["y"], what=f"token {t} alone")
    L.close()


def test_batched_decode_missing_slot_is_reported():
    wl = synth.WORKLOADS[0]
    W = synth.layer_weights(0, wl.wid, 83, wl.shape)
    L = U.layer(wl.shape, W, max_T=4)
    table = np.arange(wl.E, dtype=np.int32)
    table[:] = -1  # every expert missing: only the shared expert contributes
    x = synth.tokens(0, wl.wid, 83, 0, 4, wl.H)
    out = U.run(L, x, table=table)
    assert out["status"] == moe.MOE_ERR_SLOT
    L.close()
