"""Pins of the seeded input generator (CPU)."""
import os

import numpy as np

import synth


def _golden(root, name):
    with open(os.path.join(root, "tests", "golden", name)) as f:
        return [int(l, 16) for l in f if l.strip() and not l.startswith("#")]


def test_splitmix64_published_sequence(root):
    expected = _golden(root, "splitmix64_seed0.txt")
    assert [synth.draw(0, i) for i in range(len(expected))] == expected


def test_counter_based_and_deterministic():
    key = synth.stream_key(0, 1, 2, 3, 4)
    a = synth.uniform_u32(key, 1001)
    b = synth.uniform_u32(key, 1001)
    assert np.array_equal(a, b)
    # element i depends only on (key, i): a longer fill extends a shorter one
    c = synth.uniform_u32(key, 2000)
    assert np.array_equal(a, c[:1001])
    assert synth.stream_key(0, 1, 2, 3, 4) != synth.stream_key(0, 1, 2, 3, 5)


def test_int4_codes_uniform():
    w = synth.uniform_u32(synth.stream_key(0, 0, 0, 99, 0), 1 << 16)
    codes = ((w[:, None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF).ravel()
    counts = np.bincount(codes, minlength=16)
    expected = codes.size / 16
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 50.0  # 15 dof; p ~ 1e-5


def test_normal_and_scale_recipe():
    key = synth.stream_key(0, 0, 0, 98, 0)
    n = synth.normal_bf16(key, 200000)
    v = (n.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    s, b = synth.scale_bias(key, 50000)
    sv = (s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bv = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(sv >= 0.005 * (1 - 2 ** -8)) and np.all(bv == -8.0 * sv)
    # E|N(0,1)| = sqrt(2/pi)
    assert abs(sv.mean() - (0.005 + 0.01 * np.sqrt(2 / np.pi))) < 2e-4


def test_workload_expert_bytes():
    w = synth.WORKLOADS[2]
    assert w.expert_bytes == 1769472
    assert synth.WORKLOADS[0].expert_bytes == 30720
