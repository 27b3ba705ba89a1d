"""Pins for the oracle's acceptance from logits (readings R9-R11), CPU only.

  * exp_f32 (the specified fp32 exponential) is within 2 ulp of the exact
    exponential, exact at 0, and 0 below its range and at -inf;
  * the fp32 softmax is within a few fp32 rounding errors (scaled by the
    exponent argument) of the fp64 softmax of logits / T, for several
    temperatures;
  * adding a constant to every logit (exactly, integer logits) changes no
    probability bit;
  * the oracle's Philox equals synth's independent implementation of the
    published definition, bit for bit;
  * identical target and draft logits accept every draft (p = q);
  * the first emitted token follows the target softmax (chi-square).
"""
import numpy as np
import pytest
from scipy import stats

import synth


def test_exp_f32_is_within_two_ulp(oracle_lib):
    y = np.linspace(-85.0, 0.0, 2_000_001).astype(np.float32)
    e = oracle_lib.exp_f32(y)
    ref = np.exp(y.astype(np.float64))
    assert (np.abs(e / ref - 1.0) <= 2 * 2.0 ** -24).all()
    special = oracle_lib.exp_f32(np.array([0.0, -np.inf, -1e30, -90.0], np.float32))
    assert special[0] == 1.0 and (special[1:] == 0.0).all()


def fp64_softmax(z, T):
    z = z.astype(np.float64) / T
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


@pytest.mark.parametrize("T", [1.0, 0.7, 1.3, 0.25])
def test_softmax_close_to_fp64(oracle_lib, T):
    rng = np.random.default_rng(int(T * 100))
    B, D, V = 3, 2, 5000
    zp = (rng.standard_normal((B, D + 1, V)) * 3).astype(np.float32)
    zq = (rng.standard_normal((B, D, V)) * 3).astype(np.float32)
    p, q, _, _ = oracle_lib.logits_to_probs(zp, zq, T, 5)
    for got, z in ((p, zp), (q, zq)):
        ref = fp64_softmax(z, T)
        # the fp32 exponent argument (z - max) / T carries a relative rounding
        # error of ~2^-24, i.e. an absolute one of ~2^-24 |y|: the relative
        # error of a probability grows with how far its logit is below the max
        y = (z.astype(np.float64) - z.max(axis=-1, keepdims=True)) / T
        big = ref > 1e-30
        assert (np.abs(got[big] / ref[big] - 1) <= 1.5e-7 * (1 + np.abs(y[big]))).all()
        assert np.abs(got[ref > 1e-4] / ref[ref > 1e-4] - 1).max() < 2e-6
        assert np.abs(got.sum(axis=-1) - 1).max() < 1e-5


def test_constant_shift_changes_nothing(oracle_lib):
    rng = np.random.default_rng(0)
    zp = rng.integers(-40, 40, size=(2, 3, 700)).astype(np.float32)
    zq = rng.integers(-40, 40, size=(2, 2, 700)).astype(np.float32)
    a = oracle_lib.logits_to_probs(zp, zq, 0.9, 1)
    b = oracle_lib.logits_to_probs(zp + 1024.0, zq - 512.0, 0.9, 1)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


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
    expect = fp64_softmax(zt, T) * B
    assert stats.chisquare(counts, expect).pvalue > 1e-3


def test_row_stats_max_and_exact_sum(oracle_lib):
    """m is the row maximum (numpy's); zf is the sum of the fp32
    exponentials truncated to 2^-55, within the exponential's 2 ulp of the
    fp64 sum of exp((z - m) / T) (the truncation adds at most V 2^-55)."""
    rng = np.random.default_rng(11)
    B, D, V, T = 4, 3, 6000, 0.8
    zp = (rng.standard_normal((B, D + 1, V)) * 3).astype(np.float32)
    zq = (rng.standard_normal((B, D, V)) * 3).astype(np.float32)
    m, zf = oracle_lib.logits_row_stats(zp, zq, T)
    rows = np.concatenate([zp, zq], axis=1)
    assert np.array_equal(m, rows.max(axis=-1))
    invT = np.float32(1.0) / np.float32(T)
    y = (rows - rows.max(axis=-1, keepdims=True)) * invT          # fp32, as specified
    ref = np.exp(y.astype(np.float64)).sum(axis=-1)
    assert (np.abs(zf / ref - 1) <= 2 * 2.0 ** -24 + 2.0 ** -24 + V * 2.0 ** -55).all()
    # the maximum contributes exactly 1, so zf >= 1
    assert (zf >= 1.0).all()


def test_row_stats_truncation_is_exact_on_dyadic_rows(oracle_lib):
    """Rows whose exponentials are exactly 1 or 0 (k equal maxima, the rest
    -inf) sum without rounding: zf = k exactly and p = fl32(1 / k)."""
    V = 100
    for k in (1, 2, 3, 7, 64, 100):
        z = np.full((1, 1, V), -np.inf, np.float32)
        z[0, 0, :k] = 5.0
        m, zf = oracle_lib.logits_row_stats(z, np.zeros((1, 0, V), np.float32), 1.0)
        assert m[0, 0] == 5.0 and zf[0, 0] == np.float32(k)
        p, _, _, _ = oracle_lib.logits_to_probs(z, np.zeros((1, 0, V), np.float32), 1.0, 0)
        assert (p[0, 0, :k] == np.float32(1.0) / np.float32(k)).all() and (p[0, 0, k:] == 0).all()


def test_rows_without_a_softmax(oracle_lib):
    V = 50
    zp = np.zeros((3, 1, V), np.float32)
    zp[0, 0, 3] = np.nan
    zp[1, 0, :] = -np.inf
    zp[2, 0, 7] = np.inf
    m, zf = oracle_lib.logits_row_stats(zp, np.zeros((3, 0, V), np.float32), 1.0)
    assert (m == 0).all() and np.isinf(zf).all()
    p, _, _, _ = oracle_lib.logits_to_probs(zp, np.zeros((3, 0, V), np.float32), 1.0, 0)
    assert (p == 0).all()
