"""Pins for the oracle's accept/reject rules (CPU only).

What fixes the answer here, independently of the oracle's code:
  * greedy: a toy target model; for every possible draft sequence the
    emitted tokens must equal plain greedy decoding of that model
    ("speculative decoding produces the same output as standard decoding",
    co-design blog, "What is speculative decoding").
  * one-hot p and q turn the stochastic rule into the greedy rule.
  * exact enumeration: integrating over the uniforms interval by interval,
    the law of the emitted sequence equals the target model's own
    autoregressive law, whatever q is (llm-digest, "Math intuition").
  * the accepted-length law with per-position acceptance exactly alpha is
    truncated geometric with mean tau = (1 - alpha^(gamma+1)) / (1 - alpha)
    (LLM inference handbook, "Key metrics").
  * a chi-square test that the first emitted token follows p.
  * AL = n_acc + 1 lies in [1, 1 + D] ("What is speculative decoding").
"""
import itertools

import numpy as np
import pytest
from scipy import stats

import synth

V_TOY = 3


def dyadic_rows(rng, n_rows, V, denom_bits=10, min_weight=1):
    """Random probability rows whose entries are integers / 2^k (exact in
    fp32, and summing to exactly 1)."""
    total = 1 << denom_bits
    rows = []
    for _ in range(n_rows):
        cuts = np.sort(rng.choice(np.arange(1, total), size=V - 1, replace=False))
        w = np.diff(np.concatenate([[0], cuts, [total]]))
        rows.append(w / total)
    return np.array(rows, dtype=np.float64)


class ToyModel:
    """Context-dependent target p(.|prefix) and draft q(.|prefix)."""

    def __init__(self, seed, V, depth, one_hot=False):
        self.rng = np.random.default_rng(seed)
        self.V = V
        self.p, self.q = {}, {}
        for n in range(depth + 1):
            for prefix in itertools.product(range(V), repeat=n):
                if one_hot:
                    self.p[prefix] = np.eye(V)[self.rng.integers(V)]
                    self.q[prefix] = np.eye(V)[self.rng.integers(V)]
                else:
                    self.p[prefix], self.q[prefix] = dyadic_rows(self.rng, 2, V)


def verify_rows(model, drafts, D):
    p = np.stack([model.p[tuple(drafts[:i])] for i in range(D + 1)]).astype(np.float32)
    q = np.stack([model.q[tuple(drafts[:i])] for i in range(D)]).astype(np.float32)
    if D == 0:
        q = np.zeros((0, model.V), np.float32)
    return p, q


@pytest.mark.parametrize("D", [1, 2, 3])
def test_greedy_equals_plain_greedy_decoding(oracle_lib, D):
    model = ToyModel(100 + D, V_TOY, D)
    # plain greedy decoding of the target from the empty prefix
    ref = []
    for _ in range(D + 1):
        ref.append(int(np.argmax(model.p[tuple(ref)])))
    P, dr = [], []
    for drafts in itertools.product(range(V_TOY), repeat=D):
        p, _ = verify_rows(model, list(drafts), D)
        P.append(p)
        dr.append(drafts)
    n_acc, tok = oracle_lib.accept_greedy(np.stack(P), np.array(dr, np.int32))
    for drafts, n, t in zip(dr, n_acc, tok):
        emitted = list(drafts[:n]) + [int(t)]
        assert emitted == ref[:n + 1]
        assert 0 <= n <= D
        # the accepted prefix is the longest agreeing one
        if n < D:
            assert drafts[n] != ref[n]


def test_greedy_ties_take_lowest_index(oracle_lib):
    p = np.array([[[0.25, 0.375, 0.375, 0.0], [0.5, 0.5, 0.0, 0.0]]], np.float32)
    n, t = oracle_lib.accept_greedy(p, np.array([[1]], np.int32))
    assert n[0] == 1 and t[0] == 0
    n, t = oracle_lib.accept_greedy(p, np.array([[2]], np.int32))
    assert n[0] == 0 and t[0] == 1


def test_one_hot_sample_equals_greedy(oracle_lib):
    rng = np.random.default_rng(3)
    B, D, V = 500, 4, 7
    tgt = rng.integers(V, size=(B, D + 1))
    drafts = np.where(rng.random((B, D)) < 0.7, tgt[:, :D], rng.integers(V, size=(B, D)))
    p = np.eye(V, dtype=np.float32)[tgt]
    q = np.eye(V, dtype=np.float32)[drafts]
    u_acc = rng.random((B, D)).astype(np.float32)
    u_res = rng.random(B).astype(np.float32)
    n_s, t_s, _, _ = oracle_lib.accept_sample(p, q, drafts.astype(np.int32), u_acc, u_res)
    n_g, t_g = oracle_lib.accept_greedy(p, drafts.astype(np.int32))
    assert np.array_equal(n_s, n_g) and np.array_equal(t_s, t_g)


def enumerate_branches(model, D):
    """All (drafts, uniforms) branches with exact probability weights.

    Acceptance of draft x at a position happens iff u < p(x)/q(x), so a
    uniform at a_i/2 lands in the accept interval (length a_i = min(1, p/q))
    and one at (1+a_i)/2 in the reject interval (length 1 - a_i).  The
    draw is a step function of u_res with breakpoints C(v)/Z; its interval
    midpoints carry weight r(v)/Z.
    """
    V = model.V
    rows = []
    for drafts in itertools.product(range(V), repeat=D):
        w_draft = 1.0
        for i in range(D):
            w_draft *= model.q[drafts[:i]][drafts[i]]
        if w_draft == 0.0:
            continue
        p, q = verify_rows(model, list(drafts), D)
        a = [min(1.0, float(p[i, drafts[i]]) / float(q[i, drafts[i]])) for i in range(D)]
        for j in range(D + 1):          # j = first rejected position, D = none
            w = w_draft
            u_acc = np.full(D, 0.5)
            for i in range(j):
                w *= a[i]
                u_acc[i] = a[i] / 2
            if j < D:
                w *= 1.0 - a[j]
                u_acc[j] = (1.0 + a[j]) / 2
                r = np.maximum(0.0, p[j].astype(np.float64) - q[j].astype(np.float64))
            else:
                r = p[D].astype(np.float64)
            if w == 0.0:
                continue
            Z = r.sum()
            C = np.concatenate([[0.0], np.cumsum(r)]) / Z
            for v in range(V):
                if r[v] == 0.0:
                    continue
                rows.append((drafts, p, q, u_acc.copy(), 0.5 * (C[v] + C[v + 1]),
                             w * r[v] / Z))
    return rows


@pytest.mark.parametrize("D,seed", [(1, 1), (2, 2), (2, 5), (3, 9)])
def test_exact_law_of_emitted_sequence_equals_target(oracle_lib, D, seed):
    model = ToyModel(seed, V_TOY, D)
    rows = enumerate_branches(model, D)
    drafts = np.array([r[0] for r in rows], np.int32).reshape(len(rows), D)
    p = np.stack([r[1] for r in rows])
    q = np.stack([r[2] for r in rows])
    u_acc = np.array([r[3] for r in rows], np.float64).reshape(len(rows), D)
    u_res = np.array([r[4] for r in rows], np.float64)
    # fp32 rounding moves a midpoint by < 2^-24, far less than the shortest
    # interval (1/1024 wide), so every uniform stays inside its interval
    u_res32 = u_res.astype(np.float32)
    n_acc, tok, _, fb = oracle_lib.accept_sample(p, q, drafts, u_acc.astype(np.float32),
                                                 u_res32)
    assert not fb.any()
    law = {}
    for r, n, t in zip(rows, n_acc, tok):
        y = tuple(r[0][:n]) + (int(t),)
        law[y] = law.get(y, 0.0) + r[5]
    # extend each emitted sequence with target draws to length D+1 and
    # compare with the target's own law of D+1 tokens
    for z in itertools.product(range(V_TOY), repeat=D + 1):
        target = 1.0
        for k in range(D + 1):
            target *= model.p[z[:k]][z[k]]
        ext = 0.0
        for n in range(D + 1):
            tail = 1.0
            for k in range(n + 1, D + 1):
                tail *= model.p[z[:k]][z[k]]
            ext += law.get(z[:n + 1], 0.0) * tail
        assert abs(ext - target) < 1e-12, (z, ext, target)


def tau_rows(alpha, V=16):
    """q = a r + (1-a) s, p = a r + (1-a) t with disjoint supports of s and t:
    sum_v min(p, q) = alpha exactly."""
    r = np.full(V, 1.0 / V)
    s = np.where(np.arange(V) < V // 2, 2.0 / V, 0.0)
    t = np.where(np.arange(V) >= V // 2, 2.0 / V, 0.0)
    q = alpha * r + (1 - alpha) * s
    p = alpha * r + (1 - alpha) * t
    assert np.minimum(p, q).sum() == alpha
    return p.astype(np.float32), q.astype(np.float32)


def sampled_trials(p_row, q_row, B, D, seed):
    V = p_row.shape[0]
    p = np.ascontiguousarray(np.broadcast_to(p_row, (B, D + 1, V)))
    q = np.ascontiguousarray(np.broadcast_to(q_row, (B, D, V)))
    b = np.arange(B, dtype=np.uint64)
    i = np.arange(D, dtype=np.uint64)
    ud = synth.philox_uniform(seed, b[:, None], i[None, :], synth.STREAM_DRAFT)
    drafts = synth.draw_from_rows(q, ud)
    u_acc, u_res = synth.acceptance_uniforms(seed, B, D)
    return p, q, drafts, u_acc, u_res


@pytest.mark.parametrize("alpha,D", [(0.5, 3), (0.75, 7), (0.75, 3), (0.25, 5)])
def test_tau_closed_form(oracle_lib, alpha, D):
    B = 200_000
    p_row, q_row = tau_rows(alpha)
    p, q, drafts, u_acc, u_res = sampled_trials(p_row, q_row, B, D, seed=77)
    n_acc, _, _, _ = oracle_lib.accept_sample(p, q, drafts, u_acc, u_res)
    AL = n_acc.astype(np.float64) + 1
    assert AL.min() >= 1 and AL.max() <= D + 1
    tau = (1 - alpha ** (D + 1)) / (1 - alpha)
    law = np.array([alpha ** (k - 1) * (1 - alpha) for k in range(1, D + 1)] + [alpha ** D])
    sd = np.sqrt(((np.arange(1, D + 2) - tau) ** 2 * law).sum())
    assert abs(AL.mean() - tau) < 4 * sd / np.sqrt(B), (AL.mean(), tau)
    counts = np.bincount(n_acc, minlength=D + 1)
    chi2 = ((counts - B * law) ** 2 / (B * law)).sum()
    assert stats.chi2.sf(chi2, D) > 1e-3


@pytest.mark.parametrize("V,D,seed", [(8, 2, 21), (16, 4, 22)])
def test_first_token_follows_p_chi_square(oracle_lib, V, D, seed):
    rng = np.random.default_rng(seed)
    p_row, q_row = dyadic_rows(rng, 2, V, denom_bits=12)
    B = 300_000
    p, q, drafts, u_acc, u_res = sampled_trials(p_row.astype(np.float32),
                                                q_row.astype(np.float32), B, D, seed)
    n_acc, tok, _, _ = oracle_lib.accept_sample(p, q, drafts, u_acc, u_res)
    first = np.where(n_acc >= 1, drafts[:, 0], tok)
    counts = np.bincount(first, minlength=V)
    expect = B * p_row
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert stats.chi2.sf(chi2, V - 1) > 1e-3
    # and a distorted target (the draft itself) must be rejected by the test
    chi2_q = ((counts - B * q_row) ** 2 / (B * q_row)).sum()
    assert stats.chi2.sf(chi2_q, V - 1) < 1e-6


def test_accepted_length_range_on_random_inputs(oracle_lib):
    inp = synth.accept_inputs(5, 64, 5, 300, target_std=2.0, draft_noise=0.5)
    n, t, margin, fb = oracle_lib.accept_sample(inp["p"], inp["q"], inp["draft"], inp["u_acc"],
                                                inp["u_res"])
    assert n.min() >= 0 and n.max() <= 5
    assert t.min() >= 0 and t.max() < 300
    assert (margin >= 0).all()


def test_zero_residual_falls_back_to_target_row(oracle_lib):
    # p <= q everywhere with sum p < sum q: a rejection leaves Z = 0.
    p = np.array([[[0.25, 0.25, 0.25, 0.125], [0.25, 0.25, 0.25, 0.25]]], np.float32)
    q = np.array([[[0.25, 0.25, 0.25, 0.25]]], np.float32)
    u_acc = np.array([[0.9]], np.float32)   # 0.9 * 0.25 >= 0.125: reject
    for u, expect in [(0.1, 0), (0.5, 1), (0.95, 3)]:
        n, t, _, fb = oracle_lib.accept_sample(p, q, np.array([[3]], np.int32), u_acc,
                                               np.array([u], np.float32))
        assert n[0] == 0 and fb[0] == 1 and t[0] == expect


def test_accept_boundary_is_strict(oracle_lib):
    # u * q == p exactly must reject (strict test); just below accepts.
    p = np.array([[[0.25, 0.75], [0.5, 0.5]]], np.float32)
    q = np.array([[[0.5, 0.5]]], np.float32)
    n, _, _, _ = oracle_lib.accept_sample(p, q, np.array([[0]], np.int32),
                                          np.array([[0.5]], np.float32),
                                          np.array([0.3], np.float32))
    assert n[0] == 0
    n, _, _, _ = oracle_lib.accept_sample(p, q, np.array([[0]], np.int32),
                                          np.array([[np.nextafter(np.float32(0.5), np.float32(0))]],
                                                   np.float32),
                                          np.array([0.3], np.float32))
    assert n[0] == 1


def test_residual_draw_uses_strict_cdf_crossing(oracle_lib):
    # residual r = max(0, p - q) = [0, 0.25, 0.25, 0]: Z = 0.5.
    p = np.array([[[0.25, 0.5, 0.25, 0.0], [0.25, 0.25, 0.25, 0.25]]], np.float32)
    q = np.array([[[0.5, 0.25, 0.0, 0.25]]], np.float32)
    u_acc = np.array([[0.99]], np.float32)   # draft 0: p/q = 0.5 -> reject
    for u, expect in [(0.0, 1), (0.49, 1), (0.5, 2), (0.99, 2)]:
        n, t, _, _ = oracle_lib.accept_sample(p, q, np.array([[0]], np.int32), u_acc,
                                              np.array([u], np.float32))
        assert n[0] == 0 and t[0] == expect, (u, t[0])


# ---------------------------------------------------------------- margins
# The margin decides which GPU/oracle disagreements are exempt: per sequence,
# the smallest distance of a uniform from its decision boundary -- |u - p/q|
# for every accept test taken, and |u_res Z - C(v)| / Z for the draw (C the
# running sum, Z the total).  Dyadic rows and uniforms make every distance
# exact in fp64, so the pins compare for equality.
def _one(p_rows, q_row, x, ua, ur):
    p = np.array([p_rows], np.float32)
    q = np.array([[q_row]], np.float32)
    return (p, q, np.array([[x]], np.int32), np.array([[ua]], np.float32), np.array([ur], np.float32))


P_MARGIN = [[0.5, 0.125, 0.25, 0.125], [0.25, 0.25, 0.25, 0.25]]
Q_MARGIN = [0.25, 0.25, 0.25, 0.25]


def test_margin_of_a_rejecting_accept_test(oracle_lib):
    """Draft 1 has p/q = 1/2; u = 1/2 + 2^-12 rejects it, 2^-12 from the
    boundary.  The residual max(0, p - q) = (1/4, 0, 0, 0) has a single
    boundary, at the end: with u_res = 1/2 the draw is 1/2 from it."""
    n, t, m, _ = oracle_lib.accept_sample(*_one(P_MARGIN, Q_MARGIN, 1, 0.5 + 2.0 ** -12, 0.5))
    assert n[0] == 0 and t[0] == 0
    assert m[0] == 2.0 ** -12
    # the test far from its boundary (u = 3/4, 1/4 away) and the draw close
    # to the residual's end: u_res = 1 - 2^-10 is 2^-10 from it in units of
    # Z (Z = 1/4, so 2^-12 in absolute terms)
    n, t, m, _ = oracle_lib.accept_sample(*_one(P_MARGIN, Q_MARGIN, 1, 0.75, 1.0 - 2.0 ** -10))
    assert n[0] == 0 and t[0] == 0
    assert m[0] == 2.0 ** -10


def test_margin_of_a_draw_close_to_a_step(oracle_lib):
    """The same test accepted 2^-12 below its boundary, then the bonus draw
    from the uniform row p_1 with u_res = 1/2 + 2^-14: the running sum steps
    at 1/4, 1/2, 3/4 and 1, so the draw is 2^-14 from the step at 1/2."""
    n, t, m, _ = oracle_lib.accept_sample(*_one(P_MARGIN, Q_MARGIN, 1, 0.5 - 2.0 ** -12, 0.5 + 2.0 ** -14))
    assert n[0] == 1 and t[0] == 2
    assert m[0] == 2.0 ** -14
    # with the draw far from every step, the accept test sets the margin
    n, t, m, _ = oracle_lib.accept_sample(*_one(P_MARGIN, Q_MARGIN, 1, 0.5 - 2.0 ** -12, 0.125))
    assert n[0] == 1 and t[0] == 0 and m[0] == 2.0 ** -12


def test_margin_ignores_a_test_with_zero_draft_mass(oracle_lib):
    """q(x) = 0 < p(x) always accepts (no boundary to be near): the margin
    comes from the draw alone (u_res = 3/8 is 1/8 from the step at 1/4)."""
    q_row = [0.5, 0.0, 0.25, 0.25]
    n, t, m, _ = oracle_lib.accept_sample(*_one(P_MARGIN, q_row, 1, 0.999, 0.375))
    assert n[0] == 1 and t[0] == 1
    assert m[0] == 0.125


def test_margin_is_the_smallest_over_several_tests(oracle_lib):
    """D = 3: three accepted tests at 2^-9, 2^-7, 2^-11 from their boundaries
    (p/q = 1/2 each), then the bonus draw 1/8 from its nearest step."""
    p = np.array([[[0.5, 0.125, 0.25, 0.125]] * 3 + [[0.25, 0.25, 0.25, 0.25]]], np.float32)
    q = np.array([[[0.25, 0.25, 0.25, 0.25]] * 3], np.float32)
    ua = np.array([[0.5 - 2.0 ** -9, 0.5 - 2.0 ** -7, 0.5 - 2.0 ** -11]], np.float32)
    n, t, m, _ = oracle_lib.accept_sample(p, q, np.array([[1, 1, 1]], np.int32), ua, np.array([0.375], np.float32))
    assert n[0] == 3 and t[0] == 1
    assert m[0] == 2.0 ** -11
