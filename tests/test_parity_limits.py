"""Parity at the edges of the supported set, against the oracle.

The other parity tests stay at 1 + D <= 16 and G(1+D) <= 512 query rows per
KV head; the entry points accept 1 + D <= 64 and G(1+D) <= 1024 (eight
128-row MMA tiles reading the same K/V stream).  These cases sit on those
limits: the longest draft with a single query head per KV head, the largest
row count reached both through D and through G, acceptance (lossless and
AdaSD) walking 63 draft rows, and draft trees of 64 nodes (full 64-bit
ancestor masks).  Tolerances as in the dedicated tests (attention max-abs 2e-2
and relative L2 1e-3; acceptance bit-exact except draws within 1e-6 of a
CDF boundary).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

MARGIN = 1e-6
# boundary disagreements over the module (checked against 1e-4 of the
# sequences compared by the last test)
TALLY = {"draws": 0, "disagree": 0}


def tally(bad):
    TALLY["draws"] += len(bad)
    TALLY["disagree"] += int(bad.sum())


@pytest.fixture(scope="module")
def sv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


def bits_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("B,Hkv,G,d,D,kv_len,page", [
    (2, 2, 1, 128, 63, [64, 700], 64),      # 1 + D = 64, kv_len = 1 + D: the whole cache is drafts
    (1, 1, 16, 128, 63, [300], 32),         # G(1+D) = 1024: eight m-tiles
    (2, 1, 32, 64, 31, [33, 513], 16),      # G(1+D) = 1024 through the group size
    (3, 2, 5, 128, 40, [41, 170, 999], 48), # 205 rows: two m-tiles, the second mostly padding
])
def test_attention_at_the_limits(sv, oracle_lib, B, Hkv, G, d, D, kv_len, page):
    import torch
    inp = synth.attention_inputs(B * 100 + D, B, Hkv, G, d, D, kv_len, page_size=page)
    lse = torch.empty((B, D + 1, Hkv * G), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sv.verify_attention(bits_dev(inp.q), bits_dev(inp.k_pages), bits_dev(inp.v_pages),
                              to_dev(inp.block_table), to_dev(inp.kv_len), D, Hkv, G, lse=lse,
                              dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, lse_ref = oracle_lib.verify_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len,
                                               D, Hkv, G, d, page)
    o = out.cpu().numpy().astype(np.float64)
    err = o - ref
    assert np.isfinite(o).all()
    assert np.abs(err).max() <= 2e-2, np.abs(err).max()
    assert np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= 2e-2


def test_beyond_the_limits_is_unsupported(sv):
    """1 + D = 65, or G(1+D) = 1040 rows: rejected on the host."""
    import torch
    from speculative_decoding_verification_attention_gb300 import SpecError
    for G, D in ((1, 64), (16, 64), (40, 25)):
        inp = synth.attention_inputs(7, 1, 1, G, 64, min(D, 63), [D + 1], page_size=16)
        q = torch.zeros((1, D + 1, G, 64), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(SpecError):
            sv.verify_attention(q, bits_dev(inp.k_pages), bits_dev(inp.v_pages),
                                to_dev(inp.block_table), to_dev(np.array([D + 1], np.int32)), D, 1, G)


@pytest.mark.parametrize("V", [1000, 40000])
def test_acceptance_walks_63_drafts(sv, oracle_lib, V):
    """D = 63 with drafts close to the target, so most sequences accept long
    prefixes (some all 63): greedy and stochastic acceptance bit-exact."""
    import torch
    B, D = 6, 63
    inp = synth.accept_inputs(300 + V % 97, B, D, V, target_std=2.0, draft_noise=0.02, mode="both")
    p = inp["p"]
    n, t = sv.accept_greedy(to_dev(p), to_dev(inp["draft_greedy"]))
    torch.cuda.synchronize()
    n_ref, t_ref = oracle_lib.accept_greedy(p, inp["draft_greedy"])
    assert np.array_equal(n.cpu().numpy(), n_ref) and np.array_equal(t.cpu().numpy(), t_ref)
    assert n_ref.max() >= 32            # long accepted prefixes are exercised
    n, t = sv.accept_sample(to_dev(p), to_dev(inp["q"]), to_dev(inp["draft"]), to_dev(inp["u_acc"]),
                            to_dev(inp["u_res"]))
    torch.cuda.synchronize()
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, inp["q"], inp["draft"], inp["u_acc"], inp["u_res"])
    bad = (n.cpu().numpy() != n_ref) | (t.cpu().numpy() != t_ref)
    assert not (bad & (margin >= MARGIN)).any()
    tally(bad)
    assert n_ref.max() >= 32


@pytest.mark.parametrize("kind", ["random", "chain", "star"])
def test_tree_attention_with_64_nodes(sv, oracle_lib, kind):
    """Draft trees of 64 nodes (the 64-bit ancestor masks are full):
    G(1+D) = 256 rows, ragged lengths down to 1 + D."""
    import torch
    B, Hkv, G, d, D, page = 3, 2, 4, 128, 63, 32
    inp = synth.attention_inputs(40 + len(kind), B, Hkv, G, d, D, [64, 130, 900], page_size=page)
    parent = synth.tree_parents(50 + len(kind), B, 1 + D, kind)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sv.verify_tree_attention(bits_dev(inp.q), bits_dev(inp.k_pages), bits_dev(inp.v_pages),
                                   to_dev(inp.block_table), to_dev(inp.kv_len), to_dev(parent), D, Hkv, G,
                                   dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, _ = oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len, parent,
                                       D, Hkv, G, d, page)
    err = out.cpu().numpy().astype(np.float64) - ref
    assert np.abs(err).max() <= 2e-2
    assert np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref)


def test_tree_greedy_with_64_nodes(sv, oracle_lib):
    """Greedy tree acceptance over random 64-node trees whose nodes mostly
    carry the target's choice after their parent (deep accepted paths)."""
    import torch
    rng = np.random.default_rng(77)
    B, D, V = 8, 63, 4099
    p = synth.accept_inputs(78, B, D, V, mode="greedy")["p"]
    parent = synth.tree_parents(79, B, 1 + D, "random")
    am = np.argmax(p, axis=2)
    tokens = rng.integers(0, V, size=(B, 1 + D)).astype(np.int32)
    hit = rng.random((B, 1 + D)) < 0.9
    for b in range(B):
        for k in range(1, 1 + D):
            if hit[b, k]:
                tokens[b, k] = am[b, parent[b, k]]
    n, t, path = sv.accept_tree_greedy(to_dev(p), to_dev(tokens), to_dev(parent))
    torch.cuda.synchronize()
    n_ref, t_ref, path_ref = oracle_lib.accept_tree_greedy(p, tokens, parent)
    assert np.array_equal(n.cpu().numpy(), n_ref)
    assert np.array_equal(t.cpu().numpy(), t_ref) and np.array_equal(path.cpu().numpy(), path_ref)
    assert n_ref.max() >= 4


def test_adasd_over_63_drafts(sv, oracle_lib):
    """AdaSD relaxed acceptance with D = 63: entropy stop at the 90th
    percentile of the draft entropies (so stops fall deep in the draft),
    Jensen-Shannon threshold at the median; statistics within their
    tolerances, decisions bit-exact except draws within the margins the
    dedicated AdaSD tests use (uniform 1e-6; a statistic within its error
    bound, 1e-5 (1 + ln V), of its threshold)."""
    import torch
    B, D, V = 12, 63, 3000
    inp = synth.accept_inputs(63, B, D, V, target_std=2.5, draft_noise=0.3, mode="sample")
    p, q = inp["p"], inp["q"]
    H_ref, JS_ref = oracle_lib.adasd_stats(p, q)
    # thresholds half-way between neighbouring statistics (none lies on one)
    hs, js = np.unique(H_ref), np.unique(JS_ref)
    k, kj = int(0.9 * (len(hs) - 1)), int(0.5 * (len(js) - 1))
    tau_h, tau_js = float((hs[k] + hs[k + 1]) / 2), float((js[kj] + js[kj + 1]) / 2)
    n, t, de, H, JS = [o.cpu().numpy() for o in sv.accept_adasd(
        to_dev(p), to_dev(q), to_dev(inp["draft"]), to_dev(inp["u_acc"]), to_dev(inp["u_res"]), tau_h, tau_js)]
    torch.cuda.synchronize()
    assert (np.abs(H - H_ref) <= 1e-5 * (1 + H_ref)).all()
    jsd, jsd_ref = JS.astype(np.float64) ** 2, JS_ref ** 2
    assert (np.abs(jsd - jsd_ref) <= 2e-6 + 1e-5 * jsd_ref).all()
    n_ref, t_ref, de_ref, mu, ms, _ = oracle_lib.accept_adasd(p, q, inp["draft"], inp["u_acc"], inp["u_res"],
                                                             tau_h, tau_js)
    close = (mu < 1e-6) | (ms < 1e-5 * (1 + np.log(V)))
    bad = (n != n_ref) | (t != t_ref) | (de != de_ref)
    assert not (bad & ~close).any()
    tally(bad)
    assert (n <= de).all() and (de <= D).all()
    assert de_ref.max() >= 8


def test_zz_boundary_disagreements_stay_below_the_cap():
    """Over every comparison of this module: at most 1e-4 of the sequences
    disagree with the oracle (each one at a draw within 1e-6 of a boundary)."""
    assert TALLY["disagree"] <= 1e-4 * max(TALLY["draws"], 1), TALLY
