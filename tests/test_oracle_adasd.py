"""Pins for the oracle's AdaSD relaxed acceptance (readings R12-R15), CPU only.

  * the entropy of a draft row equals scipy's entropy (natural log), ln k for
    a row uniform over k tokens and 0 for a one-hot row;
  * the JS distance equals scipy's jensenshannon (natural log), 0 for
    identical rows and sqrt(ln 2) for rows with disjoint support;
  * with no entropy stop (tau_H = +inf) and no relaxation (tau_JS < 0) the
    acceptance is the stochastic acceptance, decision for decision;
  * d_eff is the first position whose draft entropy exceeds tau_H (rows of
    known entropy), and tau_H below every entropy draws the first token from
    the target's first row;
  * tau_JS >= sqrt(ln 2) accepts every proposed draft;
  * with one draft and JS(p, q) <= tau_JS the first emitted token follows the
    draft distribution q (it is always accepted), with JS > tau_JS the target
    p (chi-square on both).
"""
import numpy as np
import pytest
from scipy import stats
from scipy.spatial import distance

import synth

LN2 = np.log(2.0)


def test_entropy_and_js_match_scipy(oracle_lib):
    inp = synth.accept_inputs(3, 4, 5, 3000, target_std=2.0, draft_noise=0.8, mode="sample")
    p, q = inp["p"].copy(), inp["q"].copy()
    q[0, 0, :100] = 0.0        # zero entries: 0 ln 0 = 0
    p[1, 2, 50:80] = 0.0
    p /= p.sum(axis=-1, keepdims=True)   # rows sum to 1 within fp32 rounding
    q /= q.sum(axis=-1, keepdims=True)
    H, JS = oracle_lib.adasd_stats(p, q)
    for b in range(4):
        for i in range(5):
            qq = q[b, i].astype(np.float64)
            pp = p[b, i].astype(np.float64)
            # scipy's entropy normalises its input: compare on the row as given
            ref_h = stats.entropy(qq) * qq.sum() - qq.sum() * np.log(qq.sum())
            assert H[b, i] == pytest.approx(ref_h, rel=1e-9, abs=1e-9)
            # scipy normalises its inputs; the rows sum to 1 within ~1e-7
            ref = distance.jensenshannon(pp, qq)
            assert JS[b, i] == pytest.approx(ref, rel=1e-5, abs=1e-6)


@pytest.mark.parametrize("k", [1, 2, 7, 64, 1000])
def test_entropy_of_uniform_and_js_closed_forms(oracle_lib, k):
    V = 1000
    p = np.zeros((1, 2, V), np.float32)
    q = np.zeros((1, 1, V), np.float32)
    q[0, 0, :k] = 1.0 / k
    p[0, 0, :k] = 1.0 / k
    H, JS = oracle_lib.adasd_stats(p, q)
    assert H[0, 0] == pytest.approx(np.log(k), abs=1e-6)
    assert JS[0, 0] == pytest.approx(0.0, abs=1e-6)
    # disjoint supports: JSD = ln 2
    p2 = np.zeros_like(p)
    p2[0, 0, V - 1] = 1.0
    if k < V:
        _, JS2 = oracle_lib.adasd_stats(p2, q)
        assert JS2[0, 0] == pytest.approx(np.sqrt(LN2), abs=1e-7)


def test_no_stop_no_relaxation_is_the_stochastic_acceptance(oracle_lib):
    inp = synth.accept_inputs(11, 64, 6, 2000, target_std=2.0, draft_noise=0.9, mode="sample")
    args = (inp["p"], inp["q"], inp["draft"], inp["u_acc"], inp["u_res"])
    n, t, de, _, _, _ = oracle_lib.accept_adasd(*args, np.inf, -1.0)
    n_ref, t_ref, _, _ = oracle_lib.accept_sample(*args)
    assert np.array_equal(n, n_ref) and np.array_equal(t, t_ref)
    assert (de == 6).all()


def test_entropy_stop_position(oracle_lib):
    """Draft rows uniform over k_i tokens have entropy ln k_i: d_eff is the
    first i with ln k_i > tau_H."""
    V, D = 256, 5
    ks = [[2, 4, 8, 100, 3], [50, 2, 2, 2, 2], [2, 2, 2, 2, 2]]
    B = len(ks)
    p = np.full((B, D + 1, V), 1.0 / V, np.float32)
    q = np.zeros((B, D, V), np.float32)
    for b in range(B):
        for i in range(D):
            q[b, i, :ks[b][i]] = 1.0 / ks[b][i]
    draft = np.zeros((B, D), np.int32)
    u_acc = np.zeros((B, D), np.float32)   # accept wherever p(x) > 0
    u_res = np.full(B, 0.5, np.float32)
    tau = float(np.log(10.0))
    n, t, de, _, ms, _ = oracle_lib.accept_adasd(p, q, draft, u_acc, u_res, tau, -1.0)
    assert list(de) == [3, 0, 5]
    assert list(n) == [3, 0, 5]
    # all proposed drafts accepted: the token comes from the uniform target row d_eff
    assert (t == V // 2).all()
    assert (ms > 0).all()


def test_stop_before_the_first_draft_draws_from_the_first_target_row(oracle_lib):
    inp = synth.accept_inputs(12, 32, 4, 1500, mode="sample")
    n, t, de, _, _, _ = oracle_lib.accept_adasd(inp["p"], inp["q"], inp["draft"], inp["u_acc"],
                                                inp["u_res"], -1.0, -1.0)
    assert (de == 0).all() and (n == 0).all()
    n0, t0, _, _ = oracle_lib.accept_sample(inp["p"][:, :1], inp["q"][:, :0], inp["draft"][:, :0],
                                           inp["u_acc"][:, :0], inp["u_res"])
    assert np.array_equal(t, t0)


def test_full_relaxation_accepts_every_draft(oracle_lib):
    inp = synth.accept_inputs(13, 32, 4, 1500, draft_noise=3.0, mode="sample")
    n, _, de, _, _, _ = oracle_lib.accept_adasd(inp["p"], inp["q"], inp["draft"], inp["u_acc"],
                                                inp["u_res"], np.inf, float(np.sqrt(LN2)) + 1e-3)
    assert (n == 4).all() and (de == 4).all()


@pytest.mark.parametrize("relaxed", [True, False])
def test_first_token_law(oracle_lib, relaxed):
    rng = np.random.default_rng(21)
    B, D, V = 40000, 1, 6
    zt = rng.standard_normal(V) * 1.2
    zd = zt + rng.standard_normal(V) * 1.0
    pt = np.exp(zt) / np.exp(zt).sum()
    qd = np.exp(zd) / np.exp(zd).sum()
    p = np.broadcast_to(pt.astype(np.float32), (B, D + 1, V)).copy()
    q = np.broadcast_to(qd.astype(np.float32), (B, D, V)).copy()
    H, JS = oracle_lib.adasd_stats(p[:1], q[:1])
    tau_js = JS[0, 0] + 0.01 if relaxed else JS[0, 0] - 0.01
    u_d = synth.philox_uniform(5, np.arange(B)[:, None], np.arange(D)[None, :], synth.STREAM_DRAFT)
    draft = synth.draw_from_rows(q, u_d).astype(np.int32)
    u_acc, u_res = synth.acceptance_uniforms(6, B, D)
    n, t, _, _, _, _ = oracle_lib.accept_adasd(p, q, draft, u_acc, u_res, np.inf, tau_js)
    first = np.where(n >= 1, draft[:, 0], t)
    counts = np.bincount(first, minlength=V)
    expect = (qd if relaxed else pt) * B
    assert stats.chisquare(counts, expect / expect.sum() * B).pvalue > 1e-3


# ---------------------------------------------------------------- margins
# margin_stat is the smallest distance of a decisive statistic from its
# threshold (|H - tau_H| for the entropy tests taken, |JS - tau_JS| for the
# distance tests taken); margin_u is the stochastic acceptance's margin over
# the uniform decisions and the draw.  Rows of known entropy and distance
# make the distances known in closed form.
def test_margin_stat_is_the_entropy_distance(oracle_lib):
    """One position whose draft row is uniform over 4 tokens (H = ln 4),
    tau_H above it by d: the position is not a stop, and no distance test
    is taken (the exact rule accepts: p(x) = q(x)), so margin_stat = d."""
    V = 8
    q = np.zeros((1, 1, V), np.float32)
    q[0, 0, :4] = 0.25
    p = np.concatenate([q, np.full((1, 1, V), 1.0 / V, np.float32)], axis=1)
    for d in (2.0 ** -10, 2.0 ** -14, 0.125):
        tau_h = np.float32(np.log(4.0) + d)
        n, _, de, mu, ms, _ = oracle_lib.accept_adasd(p, q, np.array([[0]], np.int32), np.array([[0.5]], np.float32),
                                                      np.array([0.0625], np.float32), float(tau_h), -1.0)
        assert de[0] == 1 and n[0] == 1
        assert ms[0] == pytest.approx(float(tau_h) - np.log(4.0), rel=1e-9, abs=1e-14)
        # |u - p/q| = 1/2 for the test; the bonus draw is 1/16 from the step at 1/8
        assert mu[0] == 0.0625


def test_margin_stat_is_the_distance_distance(oracle_lib):
    """Disjoint target and draft rows (JS = sqrt(ln 2)): the exact rule
    rejects (p(x) = 0), so the distance test decides; tau_JS below JS by d
    rejects and margin_stat = d (the entropy test, ln 2 against a far
    tau_H, is farther)."""
    V = 8
    q = np.zeros((1, 1, V), np.float32)
    q[0, 0, :2] = 0.5
    p = np.zeros((1, 2, V), np.float32)
    p[0, 0, 4:] = 0.25
    p[0, 1, :] = 1.0 / V
    js = np.sqrt(LN2)
    for d in (2.0 ** -9, 2.0 ** -13):
        tau_js = np.float32(js - d)
        n, _, de, _, ms, _ = oracle_lib.accept_adasd(p, q, np.array([[0]], np.int32), np.array([[0.5]], np.float32),
                                                     np.array([0.5], np.float32), 100.0, float(tau_js))
        assert de[0] == 1 and n[0] == 0
        assert ms[0] == pytest.approx(js - float(tau_js), rel=1e-9, abs=1e-14)
    # above JS by d: relaxed, accepted
    tau_js = np.float32(js + 2.0 ** -11)
    n, _, _, _, ms, _ = oracle_lib.accept_adasd(p, q, np.array([[0]], np.int32), np.array([[0.5]], np.float32),
                                                np.array([0.5], np.float32), 100.0, float(tau_js))
    assert n[0] == 1 and ms[0] == pytest.approx(float(tau_js) - js, rel=1e-9, abs=1e-14)
