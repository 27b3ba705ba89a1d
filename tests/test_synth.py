"""Checks of the seeded input generators (no method arithmetic lives there)."""
import numpy as np
import torch
from scipy import stats

import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1e-40, 3.0e38, 1.00390625, 1.01171875], np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_philox_uniforms_are_exact_and_uniform():
    b = np.arange(200_000, dtype=np.uint64)
    u = synth.philox_uniform(123, b, np.zeros_like(b), 0)
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0
    assert np.array_equal(np.round(u.astype(np.float64) * 2 ** 24), u.astype(np.float64) * 2 ** 24)
    counts = np.bincount((u * 64).astype(int), minlength=64)
    assert stats.chisquare(counts).pvalue > 1e-3
    # counters are independent streams: a different stream id gives other values
    u2 = synth.philox_uniform(123, b[:1000], np.zeros(1000, np.uint64), 1)
    assert not np.array_equal(u[:1000], u2)


def test_philox_is_a_bijection_of_the_counter():
    # For a fixed key Philox is a permutation of the 128-bit counter space:
    # distinct counters never collide on all four output words.
    c = np.arange(50_000, dtype=np.uint64)
    w = synth.philox4x32_10(c, 0, 0, 0, 99)
    packed = set(zip(*(x.tolist() for x in w)))
    assert len(packed) == c.size


def test_paged_layout_covers_each_page_once():
    rng = np.random.default_rng(1)
    table, P = synth.paged_layout([5, 64, 65, 1], 16, rng)
    used = table[table >= 0]
    assert sorted(used.tolist()) == list(range(P))
    assert (table[0, 1:] == -1).all() and (table[2, :5] >= 0).all()


def test_tuned_sigma_reaches_alpha():
    sig, a = synth.tune_sigma_for_alpha(0.6, 4096, rows=16)
    assert abs(a - 0.6) < 0.005 and sig > 0
