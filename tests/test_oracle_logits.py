"""Pins for the oracle's acceptance from logits (readings R9-R11), CPU only.

The oracle takes p = softmax(target logits / T) and q = softmax(draft
logits / T) in fp64 and rounds each probability to fp32, then runs the
acceptance on them.  What pins it:
  * adding a constant to every logit (integer logits, exact in fp64) changes
    no probability bit, and a temperature of 1/2 equals doubled logits;
  * k equal maxima with every other logit -inf give exactly fl32(1 / k);
  * two logits (0, a) give the logistic function 1 / (1 + e^a) (scipy's
    expit), rounded to fp32;
  * every row sums to 1 within its fp32 rounding;
  * the row statistics are the row maximum and the fp64 sum of exp((z - m)
    / T), whose logarithm is scipy's logsumexp of (z - m) / T;
  * identical target and draft logits accept every draft (p = q);
  * the first emitted token follows the target softmax (chi-square);
  * the oracle's Philox equals synth's independent implementation of the
    published definition, bit for bit;
  * rows without a softmax (NaN, +inf, all -inf) read as zeros.
"""
import numpy as np
import pytest
from scipy import special, stats

import synth


def test_constant_shift_and_temperature(oracle_lib):
    rng = np.random.default_rng(0)
    zp = rng.integers(-40, 40, size=(2, 3, 700)).astype(np.float32)
    zq = rng.integers(-40, 40, size=(2, 2, 700)).astype(np.float32)
    a = oracle_lib.logits_to_probs(zp, zq, 0.9, 1)
    b = oracle_lib.logits_to_probs(zp + 1024.0, zq - 512.0, 0.9, 1)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # T = 1/2 divides exactly: the same as doubling the logits at T = 1
    c = oracle_lib.logits_to_probs(zp, zq, 0.5, 1)
    d = oracle_lib.logits_to_probs(2 * zp, 2 * zq, 1.0, 1)
    for x, y in zip(c, d):
        assert np.array_equal(x, y)
    # a different temperature does change the probabilities
    assert not np.array_equal(a[0], oracle_lib.logits_to_probs(zp, zq, 1.0, 1)[0])


@pytest.mark.parametrize("k", [1, 2, 3, 7, 64, 100])
def test_equal_maxima(oracle_lib, k):
    V = 100
    z = np.full((1, 1, V), -np.inf, np.float32)
    z[0, 0, :k] = 5.0
    p, _, _, _ = oracle_lib.logits_to_probs(z, np.zeros((1, 0, V), np.float32), 1.0, 0)
    assert (p[0, 0, :k] == np.float32(1.0 / k)).all() and (p[0, 0, k:] == 0).all()
    m, Z = oracle_lib.logits_row_stats(z, np.zeros((1, 0, V), np.float32), 1.0)
    assert m[0, 0] == 5.0 and Z[0, 0] == k


@pytest.mark.parametrize("T", [1.0, 0.7, 1.3])
def test_two_logits_give_the_logistic_function(oracle_lib, T):
    a = np.linspace(-30, 30, 601).astype(np.float32)
    z = np.stack([np.zeros_like(a), a], axis=-1)[:, None, :]          # [n, 1, 2]
    p, _, _, _ = oracle_lib.logits_to_probs(z, np.zeros((len(a), 0, 2), np.float32), T, 0)
    T32 = float(np.float32(T))                    # the temperature argument is an fp32 value
    ref0 = special.expit(-a.astype(np.float64) / T32).astype(np.float32)   # 1 / (1 + e^(a/T))
    ref1 = special.expit(a.astype(np.float64) / T32).astype(np.float32)
    # the fp64 quotient is within a few fp64 ulp of the logistic value, so
    # its fp32 rounding agrees except where that value sits on a rounding tie
    for got, ref in ((p[:, 0, 0], ref0), (p[:, 0, 1], ref1)):
        ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
        assert ulps.max() <= 1 and (ulps == 0).mean() > 0.99


@pytest.mark.parametrize("T", [1.0, 0.7, 2.0])
def test_rows_sum_to_one_and_row_stats(oracle_lib, T):
    rng = np.random.default_rng(int(T * 10))
    B, D, V = 3, 2, 5000
    zp = (rng.standard_normal((B, D + 1, V)) * 3).astype(np.float32)
    zq = (rng.standard_normal((B, D, V)) * 3).astype(np.float32)
    p, q, _, _ = oracle_lib.logits_to_probs(zp, zq, T, 5)
    for x in (p, q):
        # each fp32 rounding moves a probability by at most half an ulp
        assert np.abs(x.astype(np.float64).sum(axis=-1) - 1).max() <= V * 2.0 ** -25
    m, Z = oracle_lib.logits_row_stats(zp, zq, T)
    rows = np.concatenate([zp, zq], axis=1)
    assert np.array_equal(m, rows.max(axis=-1))
    y = (rows.astype(np.float64) - m[..., None].astype(np.float64)) / float(np.float32(T))
    assert np.allclose(np.log(Z), special.logsumexp(y, axis=-1), rtol=0, atol=1e-12)


def test_philox_matches_the_independent_implementation(oracle_lib):
    B, D, V = 300, 7, 4
    z = np.zeros((B, D + 1, V), np.float32)
    for seed in (0, 1, 0x0123456789ABCDEF, 2 ** 63 + 5):
        _, _, u_acc, u_res = oracle_lib.logits_to_probs(z, z[:, :D], 1.0, seed)
        ua, ur = synth.acceptance_uniforms(seed, B, D)
        assert np.array_equal(u_acc, ua) and np.array_equal(u_res, ur)


def test_same_model_accepts_everything(oracle_lib):
    rng = np.random.default_rng(4)
    B, D, V = 64, 5, 300
    z = (rng.standard_normal((B, D + 1, V)) * 2).astype(np.float32)
    p, _, _, _ = oracle_lib.logits_to_probs(z, z[:, :D], 1.0, 0)
    # drafts drawn from q = p
    u = synth.philox_uniform(9, np.arange(B)[:, None], np.arange(D)[None, :], synth.STREAM_DRAFT)
    draft = synth.draw_from_rows(p[:, :D], u).astype(np.int32)
    n, _, _, _ = oracle_lib.accept_sample_logits(z, z[:, :D], draft, 1.0, 3)
    assert (n == D).all()


def test_first_token_follows_the_target(oracle_lib):
    rng = np.random.default_rng(8)
    B, D, V, T = 60000, 1, 8, 0.8
    zt = (rng.standard_normal(V) * 1.5).astype(np.float32)
    zd = (zt + rng.standard_normal(V) * 1.0).astype(np.float32)
    zp = np.broadcast_to(zt, (B, D + 1, V)).copy()
    zq = np.broadcast_to(zd, (B, D, V)).copy()
    p, q, _, _ = oracle_lib.logits_to_probs(zp[:1], zq[:1], T, 0)
    u = synth.philox_uniform(21, np.arange(B)[:, None], np.arange(D)[None, :], synth.STREAM_DRAFT)
    draft = synth.draw_from_rows(np.broadcast_to(q[0], (B, D, V)), u).astype(np.int32)
    n, tok, _, _ = oracle_lib.accept_sample_logits(zp, zq, draft, T, 77)
    first = np.where(n >= 1, draft[:, 0], tok)
    counts = np.bincount(first, minlength=V)
    expect = special.softmax(zt.astype(np.float64) / float(np.float32(T))) * B
    assert stats.chisquare(counts, expect).pvalue > 1e-3


def test_rows_without_a_softmax(oracle_lib):
    V = 50
    zp = np.zeros((3, 1, V), np.float32)
    zp[0, 0, 3] = np.nan
    zp[1, 0, :] = -np.inf
    zp[2, 0, 7] = np.inf
    m, Z = oracle_lib.logits_row_stats(zp, np.zeros((3, 0, V), np.float32), 1.0)
    assert (m == 0).all() and np.isinf(Z).all()
    p, _, _, _ = oracle_lib.logits_to_probs(zp, np.zeros((3, 0, V), np.float32), 1.0, 0)
    assert (p == 0).all()
