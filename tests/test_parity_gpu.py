"""GPU parity of the CUDA library against the CPU oracle (all through the C ABI)."""
import numpy as np
import pytest

import int4_routed_expert_decode_gb300 as moe
import synth
from oracle import moe_oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

W0 = synth.WORKLOADS[0]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_decode_gb300 import build
    build.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.init()


def _weights(wl, layer=0):
    return synth.layer_weights(0, wl.wid, layer, wl.shape, zipf_s=wl.zipf_s)


def _x(wl, T, layer=0, step=0):
    return synth.tokens(0, wl.wid, layer, step, T, wl.H)


# ------------------------------------------------------------------ tiny workload
@pytest.mark.parametrize("path", [moe.MOE_PATH_AUTO, moe.MOE_PATH_GENERAL])
def test_tiny_workload_parity(path):
    W = _weights(W0)
    x = _x(W0, W0.T)
    L = U.layer(W0.shape, W, max_T=W0.T)
    moe.moe_set_path(L.ctx, path)
    out = U.run(L, x)
    ref = O.moe_block(x, W, W0.k, W0.G)
    U.assert_parity(out, ref, what="tiny")


@pytest.mark.parametrize("T", [1, 3, 31, 64, 65, 200])
def test_tiny_shapes_ragged_token_counts(T):
    """Token counts across the decode / general boundary and several tiles."""
    W = _weights(W0, layer=1)
    x = _x(W0, T, layer=1, step=T)
    L = U.layer(W0.shape, W, max_T=256)
    ref = O.moe_block(x, W, W0.k, W0.G)
    U.assert_parity(U.run(L, x), ref, what=f"T={T}")


def test_tiny_with_zipf_prior_and_larger_k():
    shape = synth.Shape(E=16, k=5, H=256, I=64, Is=128, G=32)
    W = synth.layer_weights(0, 0, 7, shape, zipf_s=1.1)
    x = synth.tokens(0, 0, 7, 0, 40, shape.H)
    L = U.layer(shape, W, max_T=40)
    ref = O.moe_block(x, W, shape.k, shape.G)
    U.assert_parity(U.run(L, x), ref, what="zipf k=5 Is=128")


def test_group_128_and_wide_hidden():
    shape = synth.Shape(E=32, k=4, H=1024, I=256, Is=128, G=128)
    W = synth.layer_weights(0, 0, 9, shape)
    x = synth.tokens(0, 0, 9, 0, 9, shape.H)
    L = U.layer(shape, W, max_T=9)
    ref = O.moe_block(x, W, shape.k, shape.G)
    U.assert_parity(U.run(L, x), ref, what="G=128")


def test_k_equals_E_dense_mixture():
    shape = synth.Shape(E=8, k=8, H=256, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 3, shape)
    x = synth.tokens(0, 0, 3, 0, 5, shape.H)
    L = U.layer(shape, W, max_T=5)
    ref = O.moe_block(x, W, shape.k, shape.G)
    U.assert_parity(U.run(L, x), ref, what="k=E")


# ------------------------------------------------------------------ exact routing
@pytest.mark.parametrize("T", [6, 40])
def test_exact_ties_go_to_lowest_index(T):
    """Identical router rows: every logit ties; the GPU must take experts 0..k-1
    (T = 40 goes through the tiled many-token router)."""
    W = _weights(W0)
    W["router_w"] = np.repeat(W["router_w"][:1], W0.E, axis=0)
    x = _x(W0, T)
    L = U.layer(W0.shape, W, max_T=T)
    out = U.run(L, x)
    assert out["topk_idx"].tolist() == [list(range(W0.k))] * T
    ref = O.moe_block(x, W, W0.k, W0.G)
    U.assert_parity(out, ref, what="ties")


def test_near_ties_one_ulp_apart():
    """Rows equal but for one bf16 ulp: fp32 logits tie or nearly; exact order decides."""
    W = _weights(W0)
    rw = W["router_w"].copy()
    for e in range(1, W0.E):
        rw[e] = rw[0]
        rw[e, e % W0.H] ^= 1  # one ulp at a different column per expert
    W["router_w"] = rw
    x = _x(W0, 16, step=5)
    L = U.layer(W0.shape, W, max_T=16)
    ref = O.moe_block(x, W, W0.k, W0.G)
    U.assert_parity(U.run(L, x), ref, what="near ties")


@pytest.mark.parametrize("T", [12, 100])
def test_duplicate_rows_with_prior(T):
    shape = synth.Shape(E=64, k=6, H=256, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 11, shape, zipf_s=0.0)
    rw = W["router_w"]
    rw[10:20] = rw[3]
    W["router_bias"] = np.zeros(shape.E, np.float32)
    x = synth.tokens(0, 0, 11, 0, T, shape.H)
    L = U.layer(shape, W, max_T=T)
    ref = O.moe_block(x, W, shape.k, shape.G)
    U.assert_parity(U.run(L, x), ref, what="duplicate rows")


# ------------------------------------------------------------------ placement, repack, errors
def test_placement_invariance_bit_identical():
    """Experts loaded in a permuted slot order with the matching table answer identically."""
    W = _weights(W0)
    x = _x(W0, 8)
    L1 = U.layer(W0.shape, W, max_T=8)
    a = U.run(L1, x)
    rng = np.random.default_rng(0)
    order = rng.permutation(W0.E)          # slot s holds expert order[s]
    Wp = dict(W)
    Wp["experts"] = {k: np.ascontiguousarray(v[order]) for k, v in W["experts"].items()}
    table = np.empty(W0.E, np.int32)
    table[order] = np.arange(W0.E, dtype=np.int32)
    L2 = U.layer(W0.shape, Wp, max_T=8)
    b = U.run(L2, x, table=table)
    for key in ("y_bits", "topk_idx", "topk_w", "perm", "offsets"):
        assert np.array_equal(a[key], b[key]), key


def test_partial_pool_with_slot_table():
    """A pool holding only the selected experts (n_slots < E) gives the same answer."""
    W = _weights(W0)
    x = _x(W0, 4)
    ref = O.moe_block(x, W, W0.k, W0.G)
    need = sorted(set(ref["topk_idx"].ravel().tolist()))
    Wp = dict(W)
    Wp["experts"] = {k: np.ascontiguousarray(v[need]) for k, v in W["experts"].items()}
    table = np.full(W0.E, -1, np.int32)
    table[need] = np.arange(len(need), dtype=np.int32)
    L = U.layer(W0.shape, Wp, max_T=4, n_slots=len(need))
    U.assert_parity(U.run(L, x, table=table), ref, what="partial pool")


def test_repack_round_trip_bytes():
    W = _weights(W0)
    L = U.layer(W0.shape, W, max_T=1)
    for slot in (0, 7, W0.E - 1):
        back = moe.moe_read_expert(L.ctx, slot, W0.H, W0.I, W0.G)
        for key, v in back.items():
            assert np.array_equal(v, W["experts"][key][slot]), (slot, key)
    back = moe.moe_read_expert(L.ctx, -1, W0.H, W0.Is, W0.G)
    for key, v in back.items():
        assert np.array_equal(v, W["shared"][key][0]), ("shared", key)


def test_device_pointer_weights_match_host_pointer_weights():
    W = _weights(W0)
    x = _x(W0, 4)
    a = U.run(U.layer(W0.shape, W, max_T=4), x)
    b = U.run(U.layer(W0.shape, W, max_T=4, device_weights=True), x)
    assert np.array_equal(a["y_bits"], b["y_bits"])


def test_missing_slot_is_reported_not_faulted():
    W = _weights(W0)
    x = _x(W0, 4)
    L = U.layer(W0.shape, W, max_T=4)
    table = np.arange(W0.E, dtype=np.int32)
    table[:] = -1
    out = U.run(L, x, table=table)
    assert out["status"] == moe.MOE_ERR_SLOT
    # the sticky word is cleared by the read: a good call reports OK again
    out = U.run(L, x)
    assert out["status"] == moe.MOE_OK


def test_host_side_argument_errors():
    import torch
    W = _weights(W0)
    L = U.layer(W0.shape, W, max_T=4)
    x = torch.zeros((8, W0.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        L.forward(x)
    assert e.value.status == moe.MOE_ERR_NOT_RESERVED
    y = torch.zeros((4, W0.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_forward(L.ctx, y, 4, None, y, torch.zeros(8, dtype=torch.int32, device="cuda"),
                        torch.zeros(8, device="cuda"))
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    # T = 0 is a no-op
    moe.moe_forward(L.ctx, x, 0, None, y, None, None)


def test_batch_equals_single_token_calls():
    """Incremental (one token per call) vs whole batch: same experts, y within tolerance."""
    W = _weights(W0, layer=2)
    x = _x(W0, 12, layer=2)
    L = U.layer(W0.shape, W, max_T=12)
    full = U.run(L, x)
    for t in range(12):
        one = U.run(L, x[t:t + 1])
        assert np.array_equal(one["topk_idx"][0], full["topk_idx"][t])
        U.assert_y_close(one["y"][0], full["y"][t], what=f"token {t}")


# ------------------------------------------------------------------ full-size single layers
@pytest.mark.parametrize("wid", [1, 2])
def test_decode_workload_single_layer(wid):
    wl = synth.WORKLOADS[wid]
    W = _weights(wl, layer=0)
    L = U.layer(wl.shape, W, max_T=4)
    for step in range(3):
        x = _x(wl, 1, layer=0, step=step)
        ref = O.moe_block(x, W, wl.k, wl.G)
        U.assert_parity(U.run(L, x), ref, what=f"wl{wid} step{step}")


def test_batched_decode_zipf_workload():
    wl = synth.WORKLOADS[3]
    W = _weights(wl)
    x = _x(wl, wl.T)
    L = U.layer(wl.shape, W, max_T=wl.T)
    ref = O.moe_block(x, W, wl.k, wl.G)
    U.assert_parity(U.run(L, x), ref, what="batch64")


def test_prefill_zipf_workload_sampled_rows():
    """T = 4096: every index and the permutation bit-exact, y on 48 sampled tokens."""
    wl = synth.WORKLOADS[4]
    W = _weights(wl)
    x = _x(wl, wl.T)
    L = U.layer(wl.shape, W, max_T=wl.T)
    out = U.run(L, x)
    rows = np.random.default_rng(4).choice(wl.T, 48, replace=False)
    rows = sorted(rows.tolist() + [0, wl.T - 1])
    ref = O.moe_block(x, W, wl.k, wl.G, tokens=rows)
    U.assert_parity(out, ref, rows=rows, what="prefill")


# ------------------------------------------------------------------ fused single-launch decode
@pytest.mark.parametrize("wid", [0, 1, 2])
def test_fused_decode_matches_oracle(wid):
    wl = synth.WORKLOADS[wid]
    W = _weights(wl, layer=3)
    L = U.layer(wl.shape, W, max_T=1)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    for step in range(4):
        x = _x(wl, 1, layer=3, step=step)
        out = U.run(L, x)
        assert moe.moe_last_launch_count(L.ctx) == 1
        ref = O.moe_block(x, W, wl.k, wl.G)
        U.assert_parity(out, ref, what=f"fused wl{wid} step{step}")


@pytest.mark.parametrize("wid", [0, 2])
def test_fused_decode_agrees_with_general_path(wid):
    wl = synth.WORKLOADS[wid]
    W = _weights(wl, layer=5)
    Lf = U.layer(wl.shape, W, max_T=1)
    Lg = U.layer(wl.shape, W, max_T=1)
    moe.moe_set_path(Lf.ctx, moe.MOE_PATH_DECODE)
    moe.moe_set_path(Lg.ctx, moe.MOE_PATH_GENERAL)
    for step in range(3):
        x = _x(wl, 1, layer=5, step=step)
        a, b = U.run(Lf, x), U.run(Lg, x)
        for key in ("topk_idx", "perm", "offsets"):
            assert np.array_equal(a[key], b[key]), key
        assert np.max(np.abs(a["topk_w"] - b["topk_w"])) <= U.W_ABS
        U.assert_y_close(a["y"], b["y"], what="fused vs general")


def test_fused_decode_other_shapes():
    """Group 128, hidden 1024, E = 64 (list length 8), larger k; inter 192 and 768,
    whose 32-code chunk counts (6, 24) are not powers of two."""
    for shape in (synth.Shape(E=64, k=6, H=1024, I=256, Is=256, G=128),
                  synth.Shape(E=300, k=12, H=512, I=128, Is=128, G=32),
                  synth.Shape(E=32, k=4, H=512, I=192, Is=192, G=64),
                  synth.Shape(E=16, k=3, H=256, I=768, Is=768, G=64)):
        W = synth.layer_weights(0, 0, 21, shape, zipf_s=0.5)
        L = U.layer(shape, W, max_T=1)
        moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
        for step in range(3):
            x = synth.tokens(0, 0, 21, step, 1, shape.H)
            U.assert_parity(U.run(L, x), O.moe_block(x, W, shape.k, shape.G),
                            what=f"fused {shape} step{step}")


def test_fused_decode_ties_and_near_ties():
    W = _weights(W0)
    rw = W["router_w"].copy()
    rw[3] = rw[9]
    rw[5] = rw[9]
    rw[7] = rw[9]
    rw[7, 11] ^= 1
    W["router_w"] = rw
    L = U.layer(W0.shape, W, max_T=1)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    for step in range(6):
        x = _x(W0, 1, step=step)
        U.assert_parity(U.run(L, x), O.moe_block(x, W, W0.k, W0.G), what=f"ties step{step}")
    W["router_w"] = np.repeat(W["router_w"][:1], W0.E, axis=0)
    L2 = U.layer(W0.shape, W, max_T=1)
    out = U.run(L2, _x(W0, 1))
    assert out["topk_idx"].tolist() == [list(range(W0.k))]


def test_fused_decode_near_ties_across_partial_lists():
    """E = 300: the block top-k's last warp list is partial (entries 256..299 of
    256..319).  Near-tied experts spread over several warp lists, the partial one
    included, are lifted into the top-k by a prior, so their order rests on the
    bounds that every warp stores next to the lists."""
    shape = synth.Shape(E=300, k=12, H=512, I=128, Is=128, G=32)
    W = synth.layer_weights(0, 0, 25, shape)
    rw = W["router_w"].copy()
    tied = [5, 70, 140, 200, 260, 277, 299]
    for j, e in enumerate(tied):
        rw[e] = rw[tied[0]]
        if j % 2:
            rw[e, (7 * j) % shape.H] ^= 1  # one bf16 ulp at a different column
    W["router_w"] = rw
    bias = np.zeros(shape.E, np.float32)
    bias[tied] = 8.0
    W["router_bias"] = bias
    L = U.layer(shape, W, max_T=1)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    for step in range(4):
        x = synth.tokens(0, 0, 25, step, 1, shape.H)
        out = U.run(L, x)
        assert set(tied) <= set(out["topk_idx"][0].tolist())
        U.assert_parity(out, O.moe_block(x, W, shape.k, shape.G), what=f"partial lists step{step}")


@pytest.mark.parametrize("wid", [0, 2])
def test_decode_far_outlier_logit(wid):
    """A prior lifts one expert's logit far above the rest: the selection
    filter's counted bins (the top quarter of [min, max]) then hold fewer than
    k + 1 logits, every logit becomes a candidate, and the exact routine ranks
    them; the top-k stays exact and the outlier comes first."""
    wl = synth.WORKLOADS[wid]
    W = _weights(wl, layer=4)
    bias = np.zeros(wl.E, np.float32) if W.get("router_bias") is None else W["router_bias"].copy()
    bias[5] += 1000.0
    W["router_bias"] = bias
    L = U.layer(wl.shape, W, max_T=1)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    for step in range(3):
        x = _x(wl, 1, layer=4, step=step)
        out = U.run(L, x)
        assert out["topk_idx"][0][0] == 5
        U.assert_parity(out, O.moe_block(x, W, wl.k, wl.G), what=f"outlier wl{wid} step{step}")


def test_fused_decode_placement_invariance():
    wl = synth.WORKLOADS[1]
    W = _weights(wl, layer=2)
    x = _x(wl, 1, layer=2)
    a = U.run(U.layer(wl.shape, W, max_T=1), x)
    order = np.random.default_rng(3).permutation(wl.E)
    Wp = dict(W)
    Wp["experts"] = {k: np.ascontiguousarray(v[order]) for k, v in W["experts"].items()}
    table = np.empty(wl.E, np.int32)
    table[order] = np.arange(wl.E, dtype=np.int32)
    b = U.run(U.layer(wl.shape, Wp, max_T=1), x, table=table)
    for key in ("y_bits", "topk_idx", "topk_w", "perm", "offsets"):
        assert np.array_equal(a[key], b[key]), key


def test_fused_decode_missing_slot_reported():
    W = _weights(W0)
    L = U.layer(W0.shape, W, max_T=1)
    x = _x(W0, 1)
    out = U.run(L, x, table=np.full(W0.E, -1, np.int32))
    assert out["status"] == moe.MOE_ERR_SLOT
    assert U.run(L, x)["status"] == moe.MOE_OK


def test_fused_decode_bounded_wait_reports_timeout():
    """A grid barrier that waits for one CTA too many runs out (about a second);
    the status says so and the context keeps working."""
    W = _weights(W0)
    L = U.layer(W0.shape, W, max_T=1)
    x = _x(W0, 1)
    moe.moe_set_test_flags(L.ctx, moe.MOE_TEST_WAIT_TIMEOUT)
    out = U.run(L, x)
    assert out["status"] == moe.MOE_ERR_TIMEOUT
    moe.moe_set_test_flags(L.ctx, 0)
    out = U.run(L, x)
    assert out["status"] == moe.MOE_OK
    U.assert_parity(out, O.moe_block(x, W, W0.k, W0.G), what="after timeout")


def test_fused_decode_graph_replay_of_stacked_layers():
    """Several layers captured in one CUDA graph (programmatic dependent
    launches between them) give the eager results on every replay."""
    import torch
    wl = synth.WORKLOADS[1]
    nl = 3
    Ws = [_weights(wl, layer=l) for l in range(nl)]
    Ls = [U.layer(wl.shape, W, max_T=1) for W in Ws]
    xs = [torch.from_numpy(_x(wl, 1, layer=l, step=7).view(np.int16)).cuda().view(torch.bfloat16)
          for l in range(nl)]
    ys = [torch.empty((1, wl.H), dtype=torch.bfloat16, device="cuda") for _ in range(nl)]
    idx = [torch.empty((1, wl.k), dtype=torch.int32, device="cuda") for _ in range(nl)]
    ws = [torch.empty((1, wl.k), dtype=torch.float32, device="cuda") for _ in range(nl)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for l in range(nl):
            moe.moe_forward(Ls[l].ctx, xs[l], 1, None, ys[l], idx[l], ws[l], stream=s)
    s.synchronize()
    eager = [y.clone() for y in ys]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for l in range(nl):
            moe.moe_forward(Ls[l].ctx, xs[l], 1, None, ys[l], idx[l], ws[l], stream=s)
    for _ in range(5):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for l in range(nl):
            assert torch.equal(ys[l], eager[l])
    for l in range(nl):
        assert Ls[l].status() == moe.MOE_OK
        ref = O.moe_block(_x(wl, 1, layer=l, step=7), Ws[l], wl.k, wl.G)
        assert idx[l].cpu().numpy().tolist() == ref["topk_idx"].tolist()
        U.assert_y_close(U.to_f64_bf16(ys[l]), ref["y"], what=f"graph layer {l}")


def test_fused_decode_topk_fallback_on_long_tie_chain():
    """512 identical router rows: every logit ties; the exact comparison of a
    run longer than the cached one settles the order (lowest ids first)."""
    wl = synth.WORKLOADS[2]
    W = _weights(wl, layer=9)
    W["router_w"] = np.repeat(W["router_w"][:1], wl.E, axis=0)
    L = U.layer(wl.shape, W, max_T=1)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_DECODE)
    x = _x(wl, 1, layer=9)
    out = U.run(L, x)
    assert out["topk_idx"].tolist() == [list(range(wl.k))]
    ref = O.moe_block(x, W, wl.k, wl.G)
    U.assert_parity(out, ref, what="tie chain")


# ------------------------------------------------------------------ tensor-core grouped GEMMs
def _prefill_layer(shape, W, max_T, **kw):
    L = U.layer(shape, W, max_T=max_T, **kw)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_PREFILL)
    return L


@pytest.mark.parametrize("T", [1, 4, 17, 130, 300])
def test_prefill_path_tiny_ragged(T):
    """One to three 128-token tiles per expert, ragged tails, N from 16 up."""
    W = _weights(W0, layer=3)
    x = _x(W0, T, layer=3, step=T)
    L = _prefill_layer(W0.shape, W, max_T=300)
    ref = O.moe_block(x, W, W0.k, W0.G)
    U.assert_parity(U.run(L, x), ref, what=f"prefill T={T}")


def test_prefill_path_hot_experts_span_many_tiles():
    """Zipf-skewed routing: hot experts own several full tiles; I != Is."""
    shape = synth.Shape(E=16, k=5, H=256, I=64, Is=128, G=32)
    W = synth.layer_weights(0, 0, 7, shape, zipf_s=1.1)
    x = synth.tokens(0, 0, 7, 1, 700, shape.H)
    L = _prefill_layer(shape, W, max_T=700)
    ref = O.moe_block(x, W, shape.k, shape.G)
    assert np.diff(ref["offsets"]).max() > 3 * 128
    U.assert_parity(U.run(L, x), ref, what="prefill zipf")


def test_prefill_path_group_128_wide_hidden():
    shape = synth.Shape(E=32, k=4, H=1024, I=256, Is=128, G=128)
    W = synth.layer_weights(0, 0, 9, shape)
    x = synth.tokens(0, 0, 9, 2, 200, shape.H)
    L = _prefill_layer(shape, W, max_T=200)
    ref = O.moe_block(x, W, shape.k, shape.G)
    U.assert_parity(U.run(L, x), ref, what="prefill G=128")


def test_prefill_path_full_width_expert_shapes():
    """hidden 2048, inter 512, group 64 (the 35B/80B expert shapes), fewer experts."""
    shape = synth.Shape(E=64, k=8, H=2048, I=512, Is=512, G=64)
    W = synth.layer_weights(0, 0, 11, shape, zipf_s=0.8)
    x = synth.tokens(0, 0, 11, 0, 160, shape.H)
    L = _prefill_layer(shape, W, max_T=160)
    ref = O.moe_block(x, W, shape.k, shape.G)
    U.assert_parity(U.run(L, x), ref, what="prefill 2048x512")


def test_prefill_path_batched_decode_workload():
    """The 64-token Zipf(1.1) batch through the grouped GEMMs, every row checked."""
    wl = synth.WORKLOADS[3]
    W = _weights(wl)
    x = _x(wl, wl.T)
    L = _prefill_layer(wl.shape, W, max_T=wl.T)
    ref = O.moe_block(x, W, wl.k, wl.G)
    U.assert_parity(U.run(L, x), ref, what="batch64 prefill path")


def test_prefill_path_agrees_with_general_path():
    W = _weights(W0, layer=4)
    x = _x(W0, 257, layer=4)
    Lp = _prefill_layer(W0.shape, W, max_T=257)
    Lg = U.layer(W0.shape, W, max_T=257)
    moe.moe_set_path(Lg.ctx, moe.MOE_PATH_GENERAL)
    a, b = U.run(Lp, x), U.run(Lg, x)
    assert np.array_equal(a["topk_idx"], b["topk_idx"])
    assert np.array_equal(a["perm"], b["perm"])
    U.assert_y_close(a["y"], b["y"], what="prefill vs general")


def test_general_path_many_tokens():
    W = _weights(W0, layer=5)
    x = _x(W0, 200, layer=5)
    L = U.layer(W0.shape, W, max_T=200)
    moe.moe_set_path(L.ctx, moe.MOE_PATH_GENERAL)
    U.assert_parity(U.run(L, x), O.moe_block(x, W, W0.k, W0.G), what="general T=200")


def test_prefill_path_missing_slot_reported():
    W = _weights(W0)
    x = _x(W0, 100)
    L = _prefill_layer(W0.shape, W, max_T=100)
    table = np.arange(W0.E, dtype=np.int32)
    table[3] = -1
    out = U.run(L, x, table=table)
    assert out["status"] == moe.MOE_ERR_SLOT
    out = U.run(L, x)
    U.assert_parity(out, O.moe_block(x, W, W0.k, W0.G), what="after slot error")


def test_prefill_path_bounded_wait_reports_timeout():
    """The MMA issuer of each CTA waits on a phase nothing completes: the wait
    runs out, every role of the CTA leaves, the status says so, and the
    context keeps working."""
    W = _weights(W0)
    x = _x(W0, 100)
    L = _prefill_layer(W0.shape, W, max_T=100)
    moe.moe_set_test_flags(L.ctx, moe.MOE_TEST_WAIT_TIMEOUT)
    out = U.run(L, x)
    assert out["status"] == moe.MOE_ERR_TIMEOUT
    moe.moe_set_test_flags(L.ctx, 0)
    out = U.run(L, x)
    U.assert_parity(out, O.moe_block(x, W, W0.k, W0.G), what="after timeout")


def test_prefill_path_graph_replay():
    """The whole prefill sequence (router to y) captured in a CUDA graph
    matches the oracle on every replay."""
    import torch
    W = _weights(W0, layer=6)
    T = 150
    x_np = _x(W0, T, layer=6)
    L = _prefill_layer(W0.shape, W, max_T=T)
    x = torch.from_numpy(x_np.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((T, W0.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, W0.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, W0.k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.moe_forward(L.ctx, x, T, None, y, idx, w, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_forward(L.ctx, x, T, None, y, idx, w, stream=s)
    ref = O.moe_block(x_np, W, W0.k, W0.G)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert L.status() == moe.MOE_OK
        assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
        U.assert_y_close(U.to_f64_bf16(y), ref["y"], what="prefill graph")


# ------------------------------------------------------------------ tensor-core router (T >= 128)
TC_SHAPE = synth.Shape(E=256, k=8, H=512, I=128, Is=128, G=64)


def test_tc_router_parity_with_prior():
    """Approximate logits on the tensor cores, certified candidates, exact order."""
    W = synth.layer_weights(0, 0, 21, TC_SHAPE, zipf_s=0.8)
    x = synth.tokens(0, 0, 21, 0, 300, TC_SHAPE.H)
    L = U.layer(TC_SHAPE, W, max_T=300)
    ref = O.moe_block(x, W, TC_SHAPE.k, TC_SHAPE.G)
    U.assert_parity(U.run(L, x), ref, what="tc router")


def test_tc_router_duplicate_rows_tie_exactly():
    """Thirty identical router rows: their logits tie exactly; lower ids first."""
    W = synth.layer_weights(0, 0, 22, TC_SHAPE)
    rw = W["router_w"]
    rw[40:70] = rw[5]
    x = synth.tokens(0, 0, 22, 0, 130, TC_SHAPE.H)
    L = U.layer(TC_SHAPE, W, max_T=130)
    ref = O.moe_block(x, W, TC_SHAPE.k, TC_SHAPE.G)
    U.assert_parity(U.run(L, x), ref, what="tc router ties")


def test_tc_router_all_rows_equal():
    """Every expert is a candidate and every logit ties: experts 0..k-1."""
    W = synth.layer_weights(0, 0, 23, TC_SHAPE)
    W["router_w"] = np.repeat(W["router_w"][:1], TC_SHAPE.E, axis=0)
    x = synth.tokens(0, 0, 23, 0, 128, TC_SHAPE.H)
    L = U.layer(TC_SHAPE, W, max_T=128)
    out = U.run(L, x)
    assert out["topk_idx"].tolist() == [list(range(TC_SHAPE.k))] * 128
    U.assert_parity(out, O.moe_block(x, W, TC_SHAPE.k, TC_SHAPE.G), what="tc router all equal")
