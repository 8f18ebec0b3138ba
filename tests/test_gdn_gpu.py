"""GPU parity of the Gated DeltaNet recurrence kernel against the float64 oracle.

Tolerance, from the kernel's fp32 arithmetic: each token's dot products over
d_k terms carry a rounding error of at most about (d_k + 4) * 2^-24 times the
sum of the magnitudes they add; the update map S -> alpha S (I - beta k^ k^T)
has norm at most 1 for alpha, beta in [0, 1], so the errors of T tokens add
up at most linearly.  Hence, per element of the output and of the state,
    |kernel - oracle| <= 4 (d_k + 4) 2^-24 (T + 1) * scale,
with scale the largest magnitude among the state, v and the output.
"""
import numpy as np
import pytest

import int4_routed_expert_decode_gb300 as moe
import synth
from oracle import gdn_oracle as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_decode_gb300 import build
    build.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.init()


def _dev(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(q, k, v, alpha, beta, state, s, splits=None):
    """Run the kernel (optionally in several calls over token ranges);
    returns (out, state) as numpy fp32."""
    import torch
    B, T = q.shape[0], q.shape[1]
    dS = _dev(state)
    out = torch.full((B, T, s.Hv, s.dv), float("nan"), dtype=torch.float32, device="cuda")
    bounds = [0] + list(splits or []) + [T]
    for t0, t1 in zip(bounds[:-1], bounds[1:]):
        n = t1 - t0
        dq, dk_, dv_ = (_dev(np.ascontiguousarray(x[:, t0:t1])) for x in (q, k, v))
        da, db = _dev(np.ascontiguousarray(alpha[:, t0:t1])), _dev(np.ascontiguousarray(beta[:, t0:t1]))
        o = torch.empty((B, n, s.Hv, s.dv), dtype=torch.float32, device="cuda")
        moe.moe_gdn_recurrence(dq, dk_, dv_, da, db, dS, o, B, n, s.Hk, s.Hv, s.dk, s.dv)
        out[:, t0:t1] = o
    torch.cuda.synchronize()
    return out.cpu().numpy(), dS.cpu().numpy()


def _tol(s, T, *arrays):
    scale = max(1.0, *(float(np.max(np.abs(a))) for a in arrays))
    return 4 * (s.dk + 4) * 2.0 ** -24 * (T + 1) * scale


def _assert_close(got, ref, tol, what):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"{what}: max err {err.max():.3e} at {worst} > tol {tol:.3e}"


def _check(seed, B, T, s, seqs=None, **kw):
    q, k, v, a, b, S0 = synth.gdn_inputs(seed, 0, B, T, s, **kw)
    out, S = _run(q, k, v, a, b, S0, s)
    seqs = range(B) if seqs is None else seqs
    for i in seqs:
        ro, rS = G.gdn_recurrence(q[i:i + 1], k[i:i + 1], v[i:i + 1], a[i:i + 1], b[i:i + 1],
                                  S0[i:i + 1])
        tol = _tol(s, T, rS, ro, G.bf16_to_f64(v[i]), S0[i])
        _assert_close(out[i:i + 1], ro, tol, f"out seq {i} {s} T={T}")
        _assert_close(S[i:i + 1], rS, tol, f"state seq {i} {s} T={T}")
    return q, k, v, a, b, S0, out, S


@pytest.mark.parametrize("B,T,shape", [
    (1, 1, synth.GdnShape(Hk=2, Hv=4, dk=128, dv=128)),
    (3, 5, synth.GdnShape(Hk=2, Hv=4, dk=128, dv=96)),
    (2, 17, synth.GdnShape(Hk=1, Hv=3, dk=64, dv=40)),
    (2, 9, synth.GdnShape(Hk=2, Hv=2, dk=256, dv=64)),
    (1, 64, synth.GdnShape(Hk=2, Hv=4, dk=128, dv=128)),
    (4, 3, synth.GdnShape(Hk=1, Hv=2, dk=128, dv=7)),
    (1, 50, synth.GdnShape(Hk=2, Hv=4, dk=64, dv=200)),
    (2, 33, synth.GdnShape(Hk=1, Hv=1, dk=256, dv=40)),
])
def test_gdn_matches_oracle(B, T, shape):
    _check(10 + T, B, T, shape)


def test_gdn_decode_step_full_size_sampled():
    """64 sequences of the 80B-class layer (16 key heads, 32 value heads,
    d_k = d_v = 128; 256 MiB of state), one decode token: sequences sampled."""
    s = synth.GdnShape()
    _check(1, 64, 1, s, seqs=[0, 31, 63])


@pytest.mark.parametrize("T", [1, 2])
def test_gdn_rows_per_warp_variants_agree(T):
    """The row split per warp depends on the state size (1 row per warp for
    a small state; 8 for a large one at T = 1, 4 at T > 1): a small and a
    large batch hold the same sequence 0 and give it bit-identical results."""
    s = synth.GdnShape(Hk=4, Hv=8, dk=128, dv=128)
    small = _check(3, 1, T, s)
    q, k, v, a, b, S0, out1, S1 = small
    B = 40  # 40 * 8 * 128 rows
    qb, kb, vb, ab, bb, Sb = synth.gdn_inputs(3, 0, B, T, s)
    for x, y in ((qb, q), (kb, k), (vb, v), (ab, a), (bb, b), (Sb, S0)):
        x[0] = y[0]
    outB, SB = _run(qb, kb, vb, ab, bb, Sb, s)
    assert np.array_equal(outB[0], out1[0]) and np.array_equal(SB[0], S1[0])


def test_gdn_incremental_equals_whole_sequence():
    """Splitting the tokens over calls changes nothing within the multi-token
    kernel (bit-identical when every part has T > 1); parts of one token run
    the decode kernel, whose sums group differently (within the tolerance)."""
    s = synth.GdnShape(Hk=2, Hv=4, dk=128, dv=128)
    q, k, v, a, b, S0 = synth.gdn_inputs(4, 0, 2, 40, s)
    o1, S1 = _run(q, k, v, a, b, S0, s)
    o2, S2 = _run(q, k, v, a, b, S0, s, splits=[3, 19, 37])
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)
    o3, S3 = _run(q, k, v, a, b, S0, s, splits=[1, 5, 39])
    tol = _tol(s, 40, S1, o1, G.bf16_to_f64(v), S0)
    _assert_close(o3, o1.astype(np.float64), tol, "single-token parts, out")
    _assert_close(S3, S1.astype(np.float64), tol, "single-token parts, state")


def test_gdn_deterministic():
    s = synth.GdnShape(Hk=2, Hv=4, dk=64, dv=64)
    q, k, v, a, b, S0 = synth.gdn_inputs(5, 0, 3, 6, s)
    o1, S1 = _run(q, k, v, a, b, S0, s)
    o2, S2 = _run(q, k, v, a, b, S0, s)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_gdn_special_gates():
    """alpha = 0 forgets the state; beta = 0 only decays it; alpha = beta = 1."""
    s = synth.GdnShape(Hk=1, Hv=2, dk=128, dv=32)
    q, k, v, a, b, S0 = synth.gdn_inputs(6, 0, 2, 4, s)
    for av, bv in ((0.0, None), (None, 0.0), (1.0, 1.0)):
        a2 = a.copy() if av is None else np.full_like(a, av)
        b2 = b.copy() if bv is None else np.full_like(b, bv)
        out, S = _run(q, k, v, a2, b2, S0, s)
        ro, rS = G.gdn_recurrence(q, k, v, a2, b2, S0)
        tol = _tol(s, 4, rS, ro, G.bf16_to_f64(v), S0)
        _assert_close(out, ro, tol, f"alpha={av} beta={bv} out")
        _assert_close(S, rS, tol, f"alpha={av} beta={bv} state")


def test_gdn_empty_calls_touch_nothing():
    import torch
    S = torch.randn(2, 4, 8, 128, device="cuda")
    before = S.clone()
    moe.moe_gdn_recurrence(None, None, None, None, None, S, None, 2, 0, 2, 4, 128, 8)
    moe.moe_gdn_recurrence(None, None, None, None, None, S, None, 0, 3, 2, 4, 128, 8)
    torch.cuda.synchronize()
    assert torch.equal(S, before)


def test_gdn_rejects_bad_arguments():
    import torch
    S = torch.zeros(1, 4, 8, 128, device="cuda")
    q = torch.zeros(1, 1, 2, 128, dtype=torch.int16, device="cuda")
    v = torch.zeros(1, 1, 4, 8, dtype=torch.int16, device="cuda")
    ab = torch.zeros(1, 1, 4, device="cuda")
    o = torch.zeros(1, 1, 4, 8, device="cuda")
    with pytest.raises(moe.MoEError) as e:  # Hv not a multiple of Hk
        moe.moe_gdn_recurrence(q, q, v, ab, ab, S, o, 1, 1, 3, 4, 128, 8)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as e:  # unsupported key dim
        moe.moe_gdn_recurrence(q, q, v, ab, ab, S, o, 1, 1, 2, 4, 96, 8)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoEError) as e:  # misaligned state
        moe.moe_gdn_recurrence(q, q, v, ab, ab, S.data_ptr() + 4, o, 1, 1, 2, 4, 128, 8)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
