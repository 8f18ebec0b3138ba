"""The tensor-core router (T >= 128) on inputs chosen to push its error margin.

The router takes approximate logits from a bf16 GEMM on the tensor cores,
keeps every expert within 2d of the k-th largest (d = 2^-10 |x| max|Wr| +
2^-22 max|prior|), certifies those, and falls back to certifying every expert
of a token whose measured error on a candidate exceeds d/8.  Each case checks
topk_idx bit for bit (and topk_w) against the C++ oracle and records the
largest observed |a - l| / (|x|_2 max_e |Wr_e|_2) over the candidates (a the
tensor-core logit, l the certified fp32 one) beside the margin 2^-10.
"""
import numpy as np
import pytest

import int4_routed_expert_decode_gb300 as moe
import synth
from oracle import cpp as C
from oracle import moe_oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

MARGIN = 2.0 ** -10


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_decode_gb300 import build
    build.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.init()


def _bits(v):
    return O.f64_to_bf16_bits(np.asarray(v, np.float64))


def _route_and_check(shape, W, x, what):
    L = U.layer(shape, W, max_T=x.shape[0])
    moe.moe_router_check_stats(L.ctx)  # start from zero
    out = U.run(L, x, want_perm=False)
    ratio, fallbacks = moe.moe_router_check_stats(L.ctx)
    assert out["status"] == moe.MOE_OK
    ref = C.moe_block(x, W, shape.k, shape.G, tokens=[0])
    assert np.array_equal(out["topk_idx"], ref["topk_idx"]), f"{what}: topk_idx differs"
    assert np.max(np.abs(out["topk_w"] - ref["topk_w"])) <= U.W_ABS, f"{what}: topk_w"
    print(f"\n{what}: max |a - l| / (|x| max|Wr|) = {ratio:.3e} "
          f"(margin 2^-10 = {MARGIN:.3e}), fallback tokens {fallbacks}")
    assert ratio < MARGIN or fallbacks > 0
    L.close()
    return ratio, fallbacks


def test_tc_router_heavy_cancellation():
    """x alternates in sign with magnitudes 1..1.5 and every router row is
    1 + small noise: each logit is a small remainder of sum|x w| ~ 1.25 H, and
    every expert falls within the filter window."""
    shape = synth.Shape(E=128, k=8, H=2048, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 60, shape)
    rng = np.random.default_rng(60)
    T = 256
    sign = np.where(np.arange(shape.H) % 2 == 0, 1.0, -1.0)
    x = _bits(sign[None, :] * (1.0 + 0.5 * rng.random((T, shape.H))))
    W["router_w"] = _bits(1.0 + 0.01 * rng.standard_normal((shape.E, shape.H)))
    _route_and_check(shape, W, x, "cancellation")


def test_tc_router_wide_exponent_range():
    """Operands spread over 2^-40 .. 2^40 with random signs: products span 160
    binades, so any alignment inside the tensor cores drops the small ones."""
    shape = synth.Shape(E=128, k=8, H=1024, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 61, shape)
    rng = np.random.default_rng(61)
    T = 192

    def spread(n):
        return (rng.choice([-1.0, 1.0], size=n) * (1.0 + rng.random(n)) *
                np.exp2(rng.integers(-40, 41, size=n)))

    x = _bits(spread(T * shape.H).reshape(T, shape.H))
    W["router_w"] = _bits(spread(shape.E * shape.H).reshape(shape.E, shape.H))
    _route_and_check(shape, W, x, "exponent range")


def test_tc_router_long_accumulation_hidden_8192():
    shape = synth.Shape(E=128, k=8, H=8192, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 62, shape)
    x = synth.tokens(0, 0, 62, 0, 128, shape.H)
    _route_and_check(shape, W, x, "H = 8192")


def test_tc_router_large_prior():
    """A prior of about 1000 on every expert (with a spread of 0.01): the fp32
    addition of the prior rounds at 6e-5, which the margin's prior term covers."""
    shape = synth.Shape(E=256, k=8, H=512, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 63, shape)
    rng = np.random.default_rng(63)
    W["router_bias"] = (1000.0 + 0.01 * rng.standard_normal(shape.E)).astype(np.float32)
    x = synth.tokens(0, 0, 63, 0, 160, shape.H)
    _route_and_check(shape, W, x, "large prior")


def test_tc_router_near_ties_in_one_element():
    """Pairs of router rows that differ by one bf16 ulp in a single element."""
    shape = synth.Shape(E=128, k=8, H=512, I=64, Is=64, G=32)
    W = synth.layer_weights(0, 0, 64, shape)
    rw = W["router_w"]
    for e in range(0, shape.E, 2):
        rw[e + 1] = rw[e]
        rw[e + 1, e % shape.H] += 1  # one ulp (same sign, finite)
    x = synth.tokens(0, 0, 64, 0, 128, shape.H)
    _route_and_check(shape, W, x, "one-ulp pairs")
