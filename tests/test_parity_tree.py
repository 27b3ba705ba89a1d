"""GPU parity of tree verification (spec_verify_tree_attention,
spec_accept_tree_greedy) against the fp64 oracle.

Attention bar as for the chain: max-abs <= 2e-2 and relative L2 <= 1e-3 on
the output and the log-sum-exp.  Acceptance is exact.  The chain tree must
reproduce the chain entry points bit for bit.
"""
import numpy as np
import pytest

import synth
from test_parity_attention import MAX_ABS, REL_L2, bits_dev, check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


def run_tree(sv, inp, parent, dev_status=None):
    import torch
    B, D, Hkv, G = inp.B, inp.D, inp.Hkv, inp.G
    lse = torch.empty((B, D + 1, Hkv * G), dtype=torch.float32, device="cuda")
    out = sv.verify_tree_attention(bits_dev(inp.q), bits_dev(inp.k_pages), bits_dev(inp.v_pages),
                                   torch.from_numpy(inp.block_table).cuda(),
                                   torch.from_numpy(inp.kv_len).cuda(),
                                   torch.from_numpy(np.ascontiguousarray(parent)).cuda(), D, Hkv, G,
                                   lse=lse, dev_status=dev_status)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


SMALL = [
    # B, Hkv, G, d, D, kv_len, page, tree
    (2, 2, 8, 128, 7, [300, 129], 64, "wide"),
    (3, 1, 8, 128, 15, [40, 200, 1000], 16, "random"),
    (2, 2, 3, 64, 9, [97, 33], 32, "star"),
    (1, 2, 32, 128, 4, [700], 64, "random"),      # G(1+D) = 160: two m-tiles
    (1, 1, 4, 64, 63, [1500], 64, "random"),      # 64 nodes: the whole mask word
    (2, 1, 16, 64, 5, [6, 4000], 80, "wide"),     # kv_len = 1 + D
    (4, 2, 4, 128, 0, [1, 64, 65, 200], 64, "chain"),
]


@pytest.mark.parametrize("B,Hkv,G,d,D,kv_len,page,kind", SMALL)
def test_tree_attention_small(sv, oracle_lib, B, Hkv, G, d, D, kv_len, page, kind):
    inp = synth.attention_inputs(61 + D, B, Hkv, G, d, D, kv_len, page_size=page)
    parent = synth.tree_parents(7 + B, B, 1 + D, kind)
    out, lse = run_tree(sv, inp, parent)
    ref, lse_ref = oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                             parent, D, Hkv, G, d, page)
    check(out, ref, lse, lse_ref)


def test_chain_tree_equals_chain_entry_point(sv):
    import torch
    from test_parity_attention import run_host_inputs
    inp = synth.attention_inputs(5, 3, 2, 8, 128, 7, [500, 130, 77], page_size=64)
    parent = synth.tree_parents(0, 3, 8, "chain")
    a, la = run_tree(sv, inp, parent)
    b, lb = run_host_inputs(sv, inp)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_malformed_tree_is_flagged(sv):
    import torch
    inp = synth.attention_inputs(6, 2, 1, 4, 64, 3, [50, 60], page_size=16)
    parent = synth.tree_parents(0, 2, 4, "chain")
    parent[1, 2] = 3                      # points forward: not topological
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = run_tree(sv, inp, parent, dev_status=st)
    assert int(st.item()) & sv.DEV_STATUS_BITS["TREE"]
    assert np.isfinite(out).all()


def test_full_step_shapes_with_a_wide_tree(sv, oracle_lib):
    """B=64 paged sequences of 4096..131072 tokens, Hkv=8, G=8, 8-node tree:
    sampled (b, h) units against the oracle, every row of each unit."""
    import torch
    lens = synth.full_step_kv_lengths(50)
    inp = synth.attention_inputs_device(71, 64, 8, 8, 128, 7, lens, page_size=64)
    parent = synth.tree_parents(3, 64, 8, "wide")
    lse = torch.empty((64, 8, 64), dtype=torch.float32, device="cuda")
    out = sv.verify_tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                   torch.from_numpy(parent).cuda(), 7, 8, 8, lse=lse)
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    bs = np.concatenate([[int(np.argmin(lens)), int(np.argmax(lens))], rng.choice(64, 4, replace=False)])
    errs, refs = [], []
    for b in bs:
        h = int(rng.integers(8))
        L = int(inp.kv_len_host[b])
        npg = (L + 63) // 64
        pages = torch.from_numpy(inp.block_table_host[b, :npg].astype(np.int64)).cuda()
        k = synth.bits_from_device(inp.k_pages[pages][:, :, h:h + 1, :].contiguous())
        v = synth.bits_from_device(inp.v_pages[pages][:, :, h:h + 1, :].contiguous())
        q = synth.bits_from_device(inp.q[b:b + 1, :, h * 8:(h + 1) * 8, :].contiguous())
        ref, lref = oracle_lib.tree_attention(q, k, v, np.arange(npg, dtype=np.int32)[None, :],
                                              np.array([L], np.int32), parent[b:b + 1], 7, 1, 8, 128, 64)
        got = out[b, :, h * 8:(h + 1) * 8, :].double().cpu().numpy()
        errs.append(got - ref[0])
        refs.append(ref[0])
    err, ref = np.concatenate(errs), np.concatenate(refs)
    assert np.abs(err).max() <= MAX_ABS
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= REL_L2
    del inp
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- acceptance
def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def tree_accept_inputs(seed, B, D, V, kind, p_match=0.7):
    """p from the synthetic acceptance inputs; node tokens drawn so that one
    child of a node often carries the target's argmax there."""
    inp = synth.accept_inputs(seed, B, D, V, mode="greedy")
    p = inp["p"]
    parent = synth.tree_parents(seed, B, 1 + D, kind)
    rng = np.random.default_rng(seed + 1)
    am = np.argmax(p, axis=2)
    tokens = rng.integers(0, V, size=(B, 1 + D)).astype(np.int32)
    for b in range(B):
        for k in range(1, 1 + D):
            if rng.random() < p_match:
                tokens[b, k] = am[b, parent[b, k]]
    return p, tokens, parent


@pytest.mark.parametrize("kind,V", [("wide", 1000), ("random", 32768), ("star", 50257),
                                    ("random", 131072), ("wide", 7)])
def test_tree_greedy_matches_oracle(sv, oracle_lib, kind, V):
    import torch
    B, D = 48, 9
    p, tokens, parent = tree_accept_inputs(17, B, D, V, kind)
    n, t, path = sv.accept_tree_greedy(to_dev(p), to_dev(tokens), to_dev(parent))
    torch.cuda.synchronize()
    n_ref, t_ref, path_ref = oracle_lib.accept_tree_greedy(p, tokens, parent)
    assert np.array_equal(n.cpu().numpy(), n_ref)
    assert np.array_equal(t.cpu().numpy(), t_ref)
    assert np.array_equal(path.cpu().numpy(), path_ref)


def test_chain_tree_acceptance_equals_greedy(sv):
    import torch
    B, D, V = 64, 7, 32768
    inp = synth.accept_inputs(23, B, D, V, mode="greedy")
    p, draft = inp["p"], inp["draft"]
    am = np.argmax(p[:, :D], axis=2)
    draft = np.where(np.random.default_rng(1).random((B, D)) < 0.8, am, draft).astype(np.int32)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), draft], axis=1)
    parent = synth.tree_parents(0, B, 1 + D, "chain")
    n1, t1, _ = sv.accept_tree_greedy(to_dev(p), to_dev(tokens), to_dev(parent))
    n2, t2 = sv.accept_greedy(to_dev(p), to_dev(draft))
    torch.cuda.synchronize()
    assert torch.equal(n1, n2) and torch.equal(t1, t2)


def test_malformed_tree_acceptance_is_flagged(sv):
    import torch
    p, tokens, parent = tree_accept_inputs(3, 4, 3, 500, "chain")
    parent[2, 0] = 0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, _ = sv.accept_tree_greedy(to_dev(p), to_dev(tokens), to_dev(parent), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sv.DEV_STATUS_BITS["TREE"]
    assert int(n[2].item()) == 0


# ---------------------------------------------------------------- stochastic
# spec_accept_tree_sample against the oracle (reading R12): n_accepted,
# token and path bit-exact, except for a sequence whose oracle margin is
# below 1e-6 (a uniform that close to a test's or a CDF step's boundary,
# where the device's fp32 working row and the oracle's fp64 one may round
# apart); such disagreements are tallied over the module and must stay at
# most 1e-4 of the sequences compared (the last test checks the tally).
SAMPLE_MARGIN = 1e-6
SAMPLE_TALLY = {"draws": 0, "disagree": 0}


def run_tree_sample(sv, inp, dev_status=None):
    import torch
    d = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
         for k in ("p", "q", "tokens", "parent", "u_acc", "u_res")}
    n, t, path = sv.accept_tree_sample(d["p"], d["q"], d["tokens"], d["parent"], d["u_acc"], d["u_res"],
                                       dev_status=dev_status)
    torch.cuda.synchronize()
    return n.cpu().numpy(), t.cpu().numpy(), path.cpu().numpy()


def check_tree_sample(sv, oracle_lib, inp):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, path = run_tree_sample(sv, inp, dev_status=st)
    n_ref, t_ref, path_ref, margin, flag = oracle_lib.accept_tree_sample(
        inp["p"], inp["q"], inp["tokens"], inp["parent"], inp["u_acc"], inp["u_res"])
    bad = (n != n_ref) | (t != t_ref) | (path != path_ref).any(axis=1)
    assert not (bad & (margin >= SAMPLE_MARGIN)).any(), np.nonzero(bad & (margin >= SAMPLE_MARGIN))
    SAMPLE_TALLY["draws"] += len(n)
    SAMPLE_TALLY["disagree"] += int(bad.sum())
    D = inp["p"].shape[1] - 1
    assert n.min() >= 0 and n.max() <= D
    for b in range(len(n)):
        assert (path[b, n[b]:] == -1).all()
        # the path is a root-to-node chain of the tree
        prev = 0
        for x in path[b, :n[b]]:
            assert inp["parent"][b, x] == prev
            prev = x
    bits = int(st.item())
    assert bits & ~0x10000 == 0, bits          # at most the zero-residual note
    return n, flag


@pytest.mark.parametrize("B,D,V,kind,noise", [(64, 7, 3000, "wide", 0.5), (48, 15, 5000, "random", 0.3),
                                               (40, 9, 2048, "star", 0.8), (30, 6, 1001, "random", 0.5),
                                               (16, 0, 700, "chain", 0.5), (20, 63, 640, "random", 0.2),
                                               (25, 5, 1, "star", 0.5), (24, 7, 10000, "wide", 0.5),
                                               (12, 5, 16383, "random", 0.4), (8, 3, 40000, "star", 0.6)])
def test_tree_sample_small(sv, oracle_lib, B, D, V, kind, noise):
    inp = synth.tree_sample_inputs(100 + D + V, B, D, V, kind=kind, draft_noise=noise)
    n, _ = check_tree_sample(sv, oracle_lib, inp)
    if D > 0 and V > 1:
        assert n.max() >= 1                     # some drafts are accepted


def test_tree_sample_chain_matches_the_chain_oracle(sv, oracle_lib):
    """On a chain the tree rule is the stochastic acceptance: the device
    tree walk agrees with the chain oracle's decisions."""
    B, D, V = 96, 7, 4096
    inp = synth.accept_inputs(5, B, D, V, mode="sample")
    T = 1 + D
    qt = np.zeros_like(inp["p"])
    qt[:, :D] = inp["q"]
    tokens = np.zeros((B, T), np.int32)
    tokens[:, 1:] = inp["draft"]
    ua = np.zeros((B, T), np.float32)
    ua[:, 1:] = inp["u_acc"]
    tree = dict(p=inp["p"], q=qt, tokens=tokens, parent=np.tile(np.arange(-1, D, dtype=np.int32), (B, 1)),
                u_acc=ua, u_res=inp["u_res"])
    n, t, path = run_tree_sample(sv, tree)
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(inp["p"], inp["q"], inp["draft"], inp["u_acc"],
                                                       inp["u_res"])
    bad = (n != n_ref) | (t != t_ref)
    assert not (bad & (margin >= SAMPLE_MARGIN)).any()
    SAMPLE_TALLY["draws"] += B
    SAMPLE_TALLY["disagree"] += int(bad.sum())


def test_tree_sample_full_size(sv, oracle_lib):
    """B = 256, D = 7, V = 131072 on the wide tree shape (up to four
    candidates per position), drafts from q at the parent."""
    inp = synth.tree_sample_inputs(2026, 256, 7, 131072, kind="wide", draft_noise=0.5)
    n, _ = check_tree_sample(sv, oracle_lib, inp)
    assert n.mean() > 0.5


def test_tree_sample_flags(sv, oracle_lib):
    import torch
    inp = synth.tree_sample_inputs(9, 4, 3, 500, kind="random")
    bad = {k: v.copy() for k, v in inp.items()}
    bad["parent"][1, 2] = 2                         # not topological
    bad["tokens"][2, 1] = 500                       # out of range
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, path = run_tree_sample(sv, bad, dev_status=st)
    bits = int(st.item())
    assert bits & sv.DEV_STATUS_BITS["TREE"] and bits & sv.DEV_STATUS_BITS["TOKEN_ID"]
    assert n[1] == 0 and n[2] == 0 and (path[1] == -1).all()
    # sequences 0 and 3 are unaffected
    n_ref, t_ref, path_ref, _, _ = oracle_lib.accept_tree_sample(inp["p"], inp["q"], inp["tokens"],
                                                                 inp["parent"], inp["u_acc"], inp["u_res"])
    for b in (0, 3):
        assert n[b] == n_ref[b] and t[b] == t_ref[b]
    # an empty residual: p = q at the root, a child on a token of zero mass
    V = 8
    p = np.zeros((1, 2, V), np.float32)
    p[0, :, :4] = 0.25
    z = dict(p=p, q=p.copy(), tokens=np.array([[0, 6]], np.int32), parent=np.array([[-1, 0]], np.int32),
             u_acc=np.array([[0, 0.5]], np.float32), u_res=np.array([0.6], np.float32))
    st.zero_()
    n, t, path = run_tree_sample(sv, z, dev_status=st)
    assert int(st.item()) & sv.DEV_STATUS_BITS["INFO_ZERO_RESIDUAL"]
    n_ref, t_ref, _, _, flag = oracle_lib.accept_tree_sample(z["p"], z["q"], z["tokens"], z["parent"],
                                                             z["u_acc"], z["u_res"])
    assert flag[0] == 1 and n[0] == n_ref[0] == 0 and t[0] == t_ref[0] == 2


def test_zz_tree_sample_disagreements_stay_below_the_cap():
    assert SAMPLE_TALLY["draws"] > 0
    assert SAMPLE_TALLY["disagree"] <= max(0, int(1e-4 * SAMPLE_TALLY["draws"])), SAMPLE_TALLY
