"""Pins for the oracle's tree verification (CPU only).

Tree attention (reading R7: a node attends to the prefix and its
root-to-node path) is checked against:
  * the chain special case, which must reproduce the (separately pinned)
    verify attention bit for bit;
  * per node, decode attention (D = 0) over a cache gathered here from the
    prefix followed by the node's path -- the meaning of the tree mask;
  * torch's fp64 scaled-dot-product attention with a materialised tree mask.
Greedy tree acceptance (reading R8) is checked against:
  * the chain special case (equals the pinned greedy acceptance);
  * a brute force over the accepted-node set on trees with distinct sibling
    tokens, written here from the definition;
  * a toy target model: the emitted tokens equal its plain greedy decoding.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import synth
from test_oracle_attention import gather_contiguous


def tree_inputs(seed, B, Hkv, G, d, D, kv_len, page, kind):
    inp = synth.attention_inputs(seed, B, Hkv, G, d, D, kv_len, page_size=page)
    parent = synth.tree_parents(seed + 1, B, 1 + D, kind)
    return inp, parent


def path_of(parent_row, k):
    path = []
    while k >= 0:
        path.append(k)
        k = int(parent_row[k])
    return path[::-1]


@pytest.mark.parametrize("B,Hkv,G,d,D,kv_len,page", [(2, 2, 3, 16, 5, [30, 41], 8),
                                                      (1, 1, 4, 32, 7, [64], 16),
                                                      (3, 2, 1, 8, 0, [3, 9, 17], 4)])
def test_chain_tree_is_verify_attention(oracle_lib, B, Hkv, G, d, D, kv_len, page):
    inp, _ = tree_inputs(7, B, Hkv, G, d, D, kv_len, page, "chain")
    parent = synth.tree_parents(0, B, 1 + D, "chain")
    a = oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                  parent, D, Hkv, G, d, page)
    b = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                    D, Hkv, G, d, page)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("kind", ["random", "star", "wide"])
def test_node_equals_decode_over_its_path(oracle_lib, kind):
    B, Hkv, G, d, D, page = 2, 2, 2, 16, 9, 8
    kv_len = [40, 23]
    inp, parent = tree_inputs(19, B, Hkv, G, d, D, kv_len, page, kind)
    out, lse = oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table,
                                         inp.kv_len, parent, D, Hkv, G, d, page)
    T = 1 + D
    for b in range(B):
        L = int(inp.kv_len[b])
        P = L - T
        for k in range(T):
            path = path_of(parent[b], k)
            keys = list(range(P)) + [P + a for a in path]
            # a one-sequence contiguous cache holding exactly those keys
            n = len(keys)
            kc = np.zeros((n, 1, Hkv, d), np.uint16)
            vc = np.zeros((n, 1, Hkv, d), np.uint16)
            j = np.asarray(keys)
            pages = inp.block_table[b, j // page]
            kc[:, 0] = inp.k_pages[pages, j % page]
            vc[:, 0] = inp.v_pages[pages, j % page]
            table = np.arange(n, dtype=np.int32)[None, :]
            qk = inp.q[b:b + 1, k:k + 1]
            o1, l1 = oracle_lib.verify_attention(qk, kc, vc, table, np.array([n], np.int32), 0,
                                                 Hkv, G, d, 1)
            np.testing.assert_allclose(out[b, k], o1[0, 0], rtol=0, atol=1e-15)
            np.testing.assert_allclose(lse[b, k], l1[0, 0], rtol=0, atol=1e-14)


def test_matches_library_sdpa_with_tree_mask(oracle_lib):
    B, Hkv, G, d, D, page = 2, 2, 3, 16, 6, 8
    inp, parent = tree_inputs(23, B, Hkv, G, d, D, [31, 50], page, "random")
    scale = 0.21
    out, _ = oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                       parent, D, Hkv, G, d, page, scale)
    q = synth.bf16_bits_to_f32(inp.q).astype(np.float64)
    T = 1 + D
    for b in range(B):
        L = int(inp.kv_len[b])
        P = L - T
        mask = np.zeros((T, L), bool)
        mask[:, :P] = True
        for k in range(T):
            for a in path_of(parent[b], k):
                mask[k, P + a] = True
        for h in range(Hkv):
            kk, vv = gather_contiguous(inp, b, h)
            qq = q[b, :, h * G:(h + 1) * G, :].reshape(T * G, d)
            m = np.repeat(mask, G, axis=0)
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(qq)[None, None], torch.from_numpy(kk)[None, None],
                torch.from_numpy(vv)[None, None], attn_mask=torch.from_numpy(m)[None, None], scale=scale)
            np.testing.assert_allclose(out[b, :, h * G:(h + 1) * G, :], o[0, 0].numpy().reshape(T, G, d),
                                       rtol=1e-12, atol=1e-12)


def test_invalid_tree_is_rejected(oracle_lib):
    inp, parent = tree_inputs(3, 1, 1, 2, 8, 3, [10], 4, "chain")
    bad = parent.copy()
    bad[0, 2] = 2                       # a node cannot be its own parent
    with pytest.raises(ValueError):
        oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len, bad,
                                  3, 1, 2, 8, 4)


# ---------------------------------------------------------------- acceptance
def test_chain_tree_acceptance_is_greedy(oracle_lib):
    B, D, V = 64, 6, 50
    inp = synth.accept_inputs(4, B, D, V, mode="greedy")
    p, draft = inp["p"], inp["draft"]
    # make some drafts agree with the target so paths get long
    am = np.argmax(p[:, :D], axis=2)
    keep = np.random.default_rng(0).random((B, D)) < 0.7
    draft = np.where(keep, am, draft).astype(np.int32)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), draft], axis=1)
    parent = synth.tree_parents(0, B, 1 + D, "chain")
    n, t, path = oracle_lib.accept_tree_greedy(p, tokens, parent)
    n_ref, t_ref = oracle_lib.accept_greedy(p, draft)
    assert np.array_equal(n, n_ref) and np.array_equal(t, t_ref)
    for b in range(B):
        assert list(path[b, :n[b]]) == list(range(1, n[b] + 1)) and (path[b, n[b]:] == -1).all()


def brute_force_tree(p, tokens, parent):
    """Deepest node whose whole root path matches the target argmax (trees
    with distinct sibling tokens have exactly one such path)."""
    T = p.shape[0]
    am = np.argmax(p.astype(np.float64), axis=1)    # lowest index of the max
    ok = np.zeros(T, bool)
    ok[0] = True
    for k in range(1, T):
        ok[k] = ok[parent[k]] and tokens[k] == am[parent[k]]
    dep = np.zeros(T, int)
    for k in range(1, T):
        dep[k] = dep[parent[k]] + 1
    best = max((k for k in range(T) if ok[k]), key=lambda k: (dep[k], -k))
    return dep[best], am[best], path_of(parent, best)[1:]


@pytest.mark.parametrize("kind", ["random", "wide", "star"])
def test_tree_acceptance_brute_force(oracle_lib, kind):
    B, D, V = 80, 9, 12
    rng = np.random.default_rng({"random": 1, "wide": 2, "star": 3}[kind])
    parent = synth.tree_parents(5, B, 1 + D, kind)
    p = rng.random((B, 1 + D, V)).astype(np.float32)
    am = np.argmax(p, axis=2)
    tokens = np.zeros((B, 1 + D), np.int32)
    for b in range(B):
        for par in range(1 + D):
            kids = [k for k in range(1, 1 + D) if parent[b, k] == par]
            # distinct sibling tokens; one of them often the target's argmax
            vals = rng.permutation(V)[:len(kids)]
            if kids and rng.random() < 0.7:
                j = rng.integers(len(kids))
                where = np.nonzero(vals == am[b, par])[0]
                if len(where):
                    vals[where[0]], vals[j] = vals[j], vals[where[0]]
                else:
                    vals[j] = am[b, par]
            tokens[b, kids] = vals
    n, t, path = oracle_lib.accept_tree_greedy(p, tokens, parent)
    for b in range(B):
        dn, dt, dpath = brute_force_tree(p[b], tokens[b], parent[b])
        assert n[b] == dn and t[b] == dt and list(path[b, :n[b]]) == dpath


def test_sibling_tie_takes_lowest_index(oracle_lib):
    V = 5
    parent = np.array([[-1, 0, 0, 2]], np.int32)
    p = np.full((1, 4, V), 0.1, np.float32)
    p[0, 0, 3] = 0.9            # target picks 3 at the root
    p[0, 2, 1] = 0.9            # below node 2 it would pick 1
    tokens = np.array([[0, 3, 3, 1]], np.int32)    # nodes 1 and 2 both carry 3
    n, t, path = oracle_lib.accept_tree_greedy(p, tokens, parent)
    assert n[0] == 1 and path[0, 0] == 1 and t[0] == int(np.argmax(p[0, 1]))


def test_emitted_tokens_are_greedy_decoding_of_a_toy_model(oracle_lib):
    """Target = a fixed toy next-token model; the draft tree holds several
    candidate continuations.  Accepted path tokens + the bonus token must be
    exactly what greedy decoding of the toy model emits."""
    V, depth, B = 6, 3, 40
    rng = np.random.default_rng(9)
    W = rng.standard_normal((V, V, V))               # logits from the last two tokens

    def model(prev2, prev1):
        z = W[prev2, prev1]
        e = np.exp(z - z.max())
        return (e / e.sum()).astype(np.float32)

    for b in range(B):
        ctx = list(rng.integers(0, V, 2))
        # a tree of all candidates of depth <= depth with 2 children per node
        parent, tokens = [-1], [ctx[-1]]
        frontier = [0]
        for _ in range(depth):
            nxt = []
            for node in frontier:
                for tok in rng.choice(V, 2, replace=False):
                    parent.append(node)
                    tokens.append(int(tok))
                    nxt.append(len(parent) - 1)
            frontier = nxt
        T = len(parent)
        seqs = {}
        for k in range(T):
            seq = [tokens[a] for a in path_of(np.array(parent), k)]
            seqs[k] = ctx[:-1] + seq
        p = np.stack([model(seqs[k][-2], seqs[k][-1]) for k in range(T)])[None]
        n, t, path = oracle_lib.accept_tree_greedy(p, np.array([tokens], np.int32),
                                                   np.array([parent], np.int32))
        emitted = [tokens[a] for a in path[0, :n[0]]] + [int(t[0])]
        # plain greedy decoding of the toy model for n + 1 steps
        s = list(ctx)
        for _ in range(n[0] + 1):
            s.append(int(np.argmax(model(s[-2], s[-1]))))
        assert emitted == s[len(ctx):]


# ---------------------------------------------------------------- stochastic
# Stochastic tree acceptance (reading R12) is checked against:
#   * the chain special case, which must reproduce the (separately pinned)
#     stochastic acceptance;
#   * hand-worked small cases with siblings (a rejected child changes the
#     row the next sibling is tested against, then the residual draw);
#   * the law of the first emitted token: with k children drafted
#     independently from q at the root, it must follow p at the root
#     exactly (the rule is lossless), checked by chi-square;
#   * the flag for an empty residual and the rejection of invalid trees.

def chain_as_tree(inp):
    """The chain acceptance's inputs laid out as a tree: node k carries draft
    k - 1 and node k's draft row is q[:, k] (the last node has none)."""
    p, q, draft, u_acc = inp["p"], inp["q"], inp["draft"], inp["u_acc"]
    B, T, V = p.shape
    D = T - 1
    qt = np.zeros_like(p)
    qt[:, :D] = q
    tokens = np.zeros((B, T), np.int32)
    tokens[:, 1:] = draft
    parent = np.tile(np.arange(-1, D, dtype=np.int32), (B, 1))
    ua = np.zeros((B, T), np.float32)
    ua[:, 1:] = u_acc
    return p, qt, tokens, parent, ua


@pytest.mark.parametrize("B,D,V", [(200, 4, 50), (60, 7, 3000), (30, 0, 100)])
def test_tree_sample_chain_equals_stochastic_acceptance(oracle_lib, B, D, V):
    inp = synth.accept_inputs(B + D, B, D, V, mode="sample")
    n, t, margin, _ = oracle_lib.accept_sample(inp["p"], inp["q"], inp["draft"], inp["u_acc"], inp["u_res"])
    p, qt, tokens, parent, ua = chain_as_tree(inp)
    n2, t2, path, margin2, flag = oracle_lib.accept_tree_sample(p, qt, tokens, parent, ua, inp["u_res"])
    # the chain draws from max(0, p - q) as it is, the tree from it divided
    # by its sum: equal except within rounding of a step
    ok = margin > 1e-9
    assert np.array_equal(n[ok], n2[ok]) and np.array_equal(t[ok], t2[ok])
    assert ok.mean() > 0.99
    for b in range(B):
        assert list(path[b, :n2[b]]) == list(range(1, n2[b] + 1))
        assert (path[b, n2[b]:] == -1).all()


def one_node_tree(p_rows, q_rows, parent, tokens, u_acc, u_res):
    p = np.asarray(p_rows, np.float32)[None]
    q = np.asarray(q_rows, np.float32)[None]
    return (p, q, np.asarray(tokens, np.int32)[None], np.asarray(parent, np.int32)[None],
            np.asarray(u_acc, np.float32)[None], np.asarray([u_res], np.float32))


def test_tree_sample_siblings_hand_worked(oracle_lib):
    # root p = (.5, .3, .2, 0), q = uniform.  Child 1 carries token 3 (p = 0:
    # rejected for any u); the working row becomes max(0, p - q) / .3 =
    # (5/6, 1/6, 0, 0).  Child 2 carries token 0: 5/6 > u * 1/4 for any u,
    # so it is accepted; child 2 is a leaf and the token is drawn from its
    # own p row (one-hot on 2).
    V = 4
    p = [[.5, .3, .2, 0], [0, 0, 0, 0], [0, 0, 1, 0]]
    q = [[.25, .25, .25, .25], [.25] * 4, [.25] * 4]
    for u in (0.0, 0.5, 0.999):
        args = one_node_tree(p, q, [-1, 0, 0], [0, 3, 0], [0, u, u], 0.3)
        n, t, path, margin, flag = oracle_lib.accept_tree_sample(*args)
        assert n[0] == 1 and path[0, 0] == 2 and t[0] == 2 and flag[0] == 0
    # child 2 carries token 1 instead: accepted iff u * 1/4 < 1/6, i.e.
    # u < 2/3.  Rejected, the row becomes max(0, (5/6, 1/6, 0, 0) - q) / sum
    # = (1, 0, 0, 0): the token is 0 whatever u_res.
    for u, acc in ((0.5, True), (0.9, False)):
        for ur in (0.0, 0.7):
            args = one_node_tree(p, q, [-1, 0, 0], [0, 3, 1], [0, 0.5, u], ur)
            n, t, path, margin, flag = oracle_lib.accept_tree_sample(*args)
            if acc:
                assert n[0] == 1 and path[0, 0] == 2
            else:
                assert n[0] == 0 and t[0] == 0 and path[0, 0] == -1
    # rejected at u = .7: the margin is the smallest of the first test's
    # |.5 - 0|, the second's |.7 - (1/6)/(1/4)| and the draw's 1 - .3
    args = one_node_tree(p, q, [-1, 0, 0], [0, 3, 1], [0, 0.5, 0.7], 0.3)
    n, _, _, margin, _ = oracle_lib.accept_tree_sample(*args)
    assert n[0] == 0 and abs(margin[0] - abs(0.7 - 2.0 / 3.0)) < 1e-6   # fp32 inputs


def test_tree_sample_empty_residual_is_flagged(oracle_lib):
    # a draft token of zero target mass is rejected even at u = 0 (0 < 0 is
    # false); the residual max(0, p - q) = (0, .3, 0) then gives token 1
    p = [[.4, .6, 0], [1, 0, 0]]
    q = [[.4, .3, .3], [1, 0, 0]]
    n, t, path, margin, flag = oracle_lib.accept_tree_sample(*one_node_tree(p, q, [-1, 0], [0, 2], [0, 0.0], 0.5))
    assert n[0] == 0 and t[0] == 1 and flag[0] == 0
    # p = q at the root and two children on a token with p = q = 0: both are
    # rejected, max(0, p - q) has no mass each time, so the row stays p and
    # the flag is set; the draw from p = (.5, .5, 0) at .75 gives token 1
    p = [[.5, .5, 0], [1, 0, 0], [1, 0, 0]]
    n, t, path, margin, flag = oracle_lib.accept_tree_sample(
        *one_node_tree(p, p, [-1, 0, 0], [0, 2, 2], [0, 0.5, 0.5], 0.75))
    assert n[0] == 0 and t[0] == 1 and flag[0] == 1


@pytest.mark.parametrize("k", [1, 3])
def test_tree_sample_first_token_follows_the_target(oracle_lib, k):
    """Root with k children drafted independently from q_0: the first token
    emitted (an accepted child's token, else the residual draw) follows p_0."""
    rng = np.random.default_rng(40 + k)
    N, V = 60000, 6
    zt = rng.standard_normal(V) * 1.5
    p0 = synth.softmax_rows_fp32(zt)
    q0 = synth.softmax_rows_fp32(zt + rng.standard_normal(V) * 1.0)
    T = 1 + k
    p = np.broadcast_to(np.concatenate([p0[None], np.tile(p0[None], (k, 1))]), (N, T, V)).copy()
    q = np.broadcast_to(np.concatenate([q0[None], np.tile(q0[None], (k, 1))]), (N, T, V)).copy()
    parent = np.tile(np.array([-1] + [0] * k, np.int32), (N, 1))
    b = np.arange(N, dtype=np.uint64)
    kk = np.arange(T, dtype=np.uint64)
    ud = synth.philox_uniform(91 + k, b[:, None], kk[None, :], synth.STREAM_DRAFT)
    tokens = np.zeros((N, T), np.int32)
    for c in range(1, T):
        tokens[:, c] = synth.draw_from_rows(np.broadcast_to(q0, (N, V)), ud[:, c])
    u_acc = synth.philox_uniform(92 + k, b[:, None], kk[None, :], synth.STREAM_ACCEPT).astype(np.float32)
    u_res = synth.philox_uniform(93 + k, b, np.zeros_like(b), synth.STREAM_RESAMPLE).astype(np.float32)
    n, t, path, _, _ = oracle_lib.accept_tree_sample(p, q, tokens, parent, u_acc, u_res)
    first = np.where(n >= 1, tokens[np.arange(N), np.maximum(path[:, 0], 0)], t)
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, p0.astype(np.float64) / p0.sum() * N).pvalue > 1e-3
    # and with more than one child, later children are accepted sometimes
    if k > 1:
        assert (path[:, 0] > 1).any()


def test_tree_sample_rejects_invalid_trees(oracle_lib):
    p = np.full((1, 3, 4), 0.25, np.float32)
    good = np.array([[-1, 0, 1]], np.int32)
    tokens = np.array([[0, 1, 2]], np.int32)
    ua = np.zeros((1, 3), np.float32)
    ur = np.zeros(1, np.float32)
    oracle_lib.accept_tree_sample(p, p, tokens, good, ua, ur)
    with pytest.raises(ValueError):
        oracle_lib.accept_tree_sample(p, p, tokens, np.array([[-1, 2, 0]], np.int32), ua, ur)
    with pytest.raises(ValueError):
        oracle_lib.accept_tree_sample(p, p, np.array([[0, 1, 4]], np.int32), good, ua, ur)
