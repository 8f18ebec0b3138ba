"""GPU parity of layer stacks: L chained blocks for one token in one launch.

Each layer is checked on exactly the input the GPU used: the residual chain
is rebuilt on the host from the GPU's own bf16 block outputs (bit-exact), the
GPU's RMSNorm output is compared with the oracle's on the same residual (one
bf16 ulp: fp32 on the GPU, fp64 in the oracle, one rounding each), and the
block is compared with the oracle on the GPU's normalised input.
"""
import numpy as np
import pytest

import int4_routed_expert_decode_gb300 as moe
import synth
from oracle import moe_oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_decode_gb300 import build
    build.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.init()


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _norm_weights(H, L, seed):
    rng = np.random.default_rng(seed)
    return [O.f64_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(H)) for _ in range(L)]


def _make(shape, Ws, g_bits, n_slots=None):
    layers = [U.layer(shape, W, max_T=1, n_slots=n_slots) for W in Ws]
    norms = None if g_bits is None else [_dev(g) for g in g_bits]
    st = moe.MoEStack(layers, norms, EPS)
    st._norm_tensors = norms  # keep the device copies alive
    return st


def _bf16_ulp(v):
    _, e = np.frexp(np.asarray(v, np.float64))
    return np.ldexp(1.0, e - 8)


def check_stack(shape, Ws, g_bits, x_bits, outs, what=""):
    """outs = (x_out, y, xn, topk_idx, topk_w) from MoEStack.forward."""
    x_out, y, xn, idx, w = outs
    L = len(Ws)
    y_bits, xn_bits = _bits(y), _bits(xn)
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    xs = [np.asarray(x_bits, np.uint16)]
    for l in range(L):
        xs.append(O.residual_add(xs[l], O.bf16_to_f64(y_bits[l])))
    assert np.array_equal(_bits(x_out), xs[L]), f"{what} residual chain"
    for l in range(L):
        g = None if g_bits is None else g_bits[l]
        ref_n = O.rms_norm(xs[l], g, EPS)
        a, b = O.bf16_to_f64(xn_bits[l]), O.bf16_to_f64(ref_n)
        diff = np.abs(a - b)
        assert np.all(diff <= _bf16_ulp(b) + 0.0), f"{what} layer {l} RMSNorm beyond one ulp"
        assert np.count_nonzero(diff) <= max(4, shape.H // 128), f"{what} layer {l} RMSNorm"
        ref = O.moe_block(xn_bits[l][None, :], Ws[l], shape.k, shape.G)
        assert idx[l].tolist() == ref["topk_idx"][0].tolist(), f"{what} layer {l} topk_idx"
        assert np.max(np.abs(w[l] - ref["topk_w"][0])) <= U.W_ABS, f"{what} layer {l} topk_w"
        U.assert_y_close(O.bf16_to_f64(y_bits[l])[None, :], ref["y"], what=f"{what} layer {l}")


def _layers(wl, n, first=0):
    return [synth.layer_weights(0, wl.wid, first + l, wl.shape, zipf_s=wl.zipf_s) for l in range(n)]


def test_stack_tiny_matches_oracle():
    wl = synth.WORKLOADS[0]
    L = 4
    Ws = _layers(wl, L)
    g = _norm_weights(wl.H, L, 1)
    st = _make(wl.shape, Ws, g)
    for step in range(3):
        x = synth.tokens(0, wl.wid, 0, step, 1, wl.H)[0]
        outs = st.forward(_dev(x))
        assert st.status() == moe.MOE_OK
        check_stack(wl.shape, Ws, g, x, outs, what=f"tiny step {step}")


def test_stack_tiny_matches_oracle_end_to_end():
    """A short stack also agrees with the oracle's own chain from x alone."""
    wl = synth.WORKLOADS[0]
    L = 3
    Ws = _layers(wl, L, first=7)
    g = _norm_weights(wl.H, L, 2)
    st = _make(wl.shape, Ws, g)
    x = synth.tokens(0, wl.wid, 7, 0, 1, wl.H)[0]
    x_out, y, xn, idx, w = st.forward(_dev(x))
    assert st.status() == moe.MOE_OK
    ref = O.moe_stack(x, Ws, g, wl.k, wl.G, EPS)
    assert idx.cpu().numpy().tolist() == ref["topk_idx"].tolist()
    U.assert_y_close(O.bf16_to_f64(_bits(y)), ref["y"], what="chain y")
    U.assert_y_close(O.bf16_to_f64(_bits(x_out))[None], O.bf16_to_f64(ref["x"][L])[None],
                     what="chain x_out")


@pytest.mark.parametrize("wid", [1, 2])
def test_stack_decode_shapes(wid):
    wl = synth.WORKLOADS[wid]
    L = 4
    Ws = _layers(wl, L, first=2)
    g = _norm_weights(wl.H, L, 3)
    st = _make(wl.shape, Ws, g)
    for step in range(2):
        x = synth.tokens(0, wl.wid, 2, step, 1, wl.H)[0]
        outs = st.forward(_dev(x))
        assert st.status() == moe.MOE_OK
        check_stack(wl.shape, Ws, g, x, outs, what=f"wl{wid} step {step}")


def test_stack_with_slot_tables_and_unit_norms():
    """Experts stored in reversed slots, one table per layer; no norm weights."""
    import torch
    wl = synth.WORKLOADS[2]
    L = 2
    Ws = _layers(wl, L, first=11)
    Wr = []
    for W in Ws:
        R = dict(W)
        R["experts"] = {k: np.ascontiguousarray(v[::-1]) for k, v in W["experts"].items()}
        Wr.append(R)
    st = _make(wl.shape, Wr, None)
    tables = torch.as_tensor(np.tile(np.arange(wl.E)[::-1], (L, 1)).astype(np.int32)).cuda()
    x = synth.tokens(0, wl.wid, 11, 0, 1, wl.H)[0]
    outs = st.forward(_dev(x), tables=tables)
    assert st.status() == moe.MOE_OK
    check_stack(wl.shape, Ws, None, x, outs, what="tables")


def test_stack_output_may_overwrite_its_input():
    import torch
    wl = synth.WORKLOADS[1]
    L = 2
    Ws = _layers(wl, L, first=5)
    st = _make(wl.shape, Ws, None)
    x = synth.tokens(0, wl.wid, 5, 0, 1, wl.H)[0]
    a = st.forward(_dev(x))
    xb = _dev(x)
    st.forward(xb, x_out=xb)
    assert st.status() == moe.MOE_OK
    assert torch.equal(a[0], xb)


def test_stack_graph_replay_matches_eager():
    import torch
    wl = synth.WORKLOADS[1]
    L = 3
    Ws = _layers(wl, L, first=30)
    g = _norm_weights(wl.H, L, 4)
    st = _make(wl.shape, Ws, g)
    x = _dev(synth.tokens(0, wl.wid, 30, 0, 1, wl.H)[0])
    bufs = [torch.empty((wl.H,), dtype=torch.bfloat16, device="cuda"),
            torch.empty((L, wl.H), dtype=torch.bfloat16, device="cuda"),
            torch.empty((L, wl.H), dtype=torch.bfloat16, device="cuda"),
            torch.empty((L, wl.k), dtype=torch.int32, device="cuda"),
            torch.empty((L, wl.k), dtype=torch.float32, device="cuda")]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st.forward(x, x_out=bufs[0], y=bufs[1], xn=bufs[2], topk_idx=bufs[3], topk_w=bufs[4],
                   stream=s)
    s.synchronize()
    eager = [b.clone() for b in bufs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st.forward(x, x_out=bufs[0], y=bufs[1], xn=bufs[2], topk_idx=bufs[3], topk_w=bufs[4],
                   stream=s)
    for _ in range(4):
        for b in bufs:
            b.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for b, e in zip(bufs, eager):
            assert torch.equal(b, e)
    assert st.status() == moe.MOE_OK


def test_stack_bounded_wait_reports_timeout_and_recovers():
    """Every layer's logits exchange waits for one arrival too many (about a
    second each); the status says so, the counters are reset, and the next
    launch is correct."""
    wl = synth.WORKLOADS[0]
    L = 2
    Ws = _layers(wl, L, first=40)
    st = _make(wl.shape, Ws, None)
    x = synth.tokens(0, wl.wid, 40, 0, 1, wl.H)[0]
    moe.moe_stack_set_test_flags(st.stack, moe.MOE_TEST_WAIT_TIMEOUT)
    st.forward(_dev(x))
    assert st.status() == moe.MOE_ERR_TIMEOUT
    moe.moe_stack_set_test_flags(st.stack, 0)
    outs = st.forward(_dev(x))
    assert st.status() == moe.MOE_OK
    check_stack(wl.shape, Ws, None, x, outs, what="after timeout")


def test_decode_graph_replays_correctly_after_a_timeout_reset():
    """The single-layer decode kernel captured in a graph: an eager launch with
    the timeout hook fails, moe_get_status resets the exchange counters, and
    the graph captured before still replays the right results."""
    import torch
    wl = synth.WORKLOADS[2]
    W = synth.layer_weights(0, wl.wid, 50, wl.shape)
    lay = U.layer(wl.shape, W, max_T=1)
    moe.moe_set_path(lay.ctx, moe.MOE_PATH_DECODE)
    x = _dev(synth.tokens(0, wl.wid, 50, 0, 1, wl.H))
    y = torch.empty((1, wl.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((1, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, wl.k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        moe.moe_forward(lay.ctx, x, 1, None, y, idx, w, stream=s)  # warm-up
    s.synchronize()
    with torch.cuda.graph(graph, stream=s):
        moe.moe_forward(lay.ctx, x, 1, None, y, idx, w, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    ref_y, ref_idx = y.clone(), idx.clone()
    moe.moe_set_test_flags(lay.ctx, moe.MOE_TEST_WAIT_TIMEOUT)
    moe.moe_forward(lay.ctx, x, 1, None, y, idx, w)
    assert lay.status() == moe.MOE_ERR_TIMEOUT
    moe.moe_set_test_flags(lay.ctx, 0)
    for _ in range(3):
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref_y) and torch.equal(idx, ref_idx)
    assert lay.status() == moe.MOE_OK
    ref = O.moe_block(synth.tokens(0, wl.wid, 50, 0, 1, wl.H), W, wl.k, wl.G)
    assert idx.cpu().numpy().tolist() == ref["topk_idx"].tolist()
