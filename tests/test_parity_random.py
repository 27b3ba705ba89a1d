"""Seeded random shapes for every entry point of the step (chain and tree
attention, GEMM, greedy, stochastic and tree acceptance, acceptance from
logits), against the oracle.

Each case draws its shape from a fixed seed inside the supported set --
group size, draft length (1 + D <= 16, G(1+D) up to 512 rows; the limits
of the supported set have their own cases in test_parity_limits.py), head_dim,
page size (multiples of 16), ragged lengths down to 1 + D; vocabulary sizes
with and without 16-byte rows; GEMM shapes with ragged M -- so that
combinations the hand-written cases do not name are still compared.  The
tolerances are the ones of the dedicated parity tests: attention max-abs
2e-2 and relative L2 1e-3, GEMM relative L2 5e-3, acceptance bit-exact
except draws within 1e-6 of a CDF boundary.
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


def attention_shape(rng):
    while True:
        G = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 32]))
        D = int(rng.integers(0, 16))
        if G * (1 + D) <= 512:
            break
    B = int(rng.integers(1, 5))
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    d = int(rng.choice([64, 128]))
    page = int(rng.choice([16, 32, 48, 64, 128]))
    lens = rng.integers(1 + D, 3000, size=B)
    lens[rng.integers(0, B)] = 1 + D + int(rng.integers(0, 3))   # one (nearly) minimal sequence
    return B, Hkv, G, d, D, lens.astype(np.int32), page


@pytest.mark.parametrize("seed", range(24))
def test_random_attention(sv, oracle_lib, seed):
    import torch
    rng = np.random.default_rng(1000 + seed)
    B, Hkv, G, d, D, lens, page = attention_shape(rng)
    inp = synth.attention_inputs(2000 + seed, B, Hkv, G, d, D, lens, page_size=page)
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
    assert np.abs(err).max() <= 2e-2, (B, Hkv, G, d, D, page, np.abs(err).max())
    assert np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref), (B, Hkv, G, d, D, page)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.abs(l - lse_ref).max() <= 2e-2


@pytest.mark.parametrize("seed", range(12))
def test_random_gemm(sv, oracle_lib, seed):
    rng = np.random.default_rng(3000 + seed)
    M = int(rng.choice([1, 3, 17, 64, 100, 200, 256, 257, 300, 511, 700, 1000]))
    N = 128 * int(rng.integers(1, 25))
    K = 64 * int(rng.integers(1, 33))
    xb, wb = synth.gemm_inputs(4000 + seed, M, N, K)
    y = sv.verify_gemm(bits_dev(xb), bits_dev(wb))
    yr = oracle_lib.gemm(xb, wb)
    e = y.float().cpu().numpy().astype(np.float64) - yr
    assert np.linalg.norm(e) <= 5e-3 * np.linalg.norm(yr), (M, N, K)


@pytest.mark.parametrize("seed", range(12))
def test_random_acceptance(sv, oracle_lib, seed):
    import torch
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(1, 40))
    D = int(rng.integers(0, 12))
    V = int(rng.choice([5, 257, 1000, 4096, 5003, 32768, 50000, 65537]))
    inp = synth.accept_inputs(6000 + seed, B, D, V, target_std=2.0, draft_noise=float(rng.uniform(0.3, 1.5)),
                              mode="both")
    p = inp["p"]
    n, t = sv.accept_greedy(to_dev(p), to_dev(inp["draft_greedy"]) if D else None)
    torch.cuda.synchronize()
    n_ref, t_ref = oracle_lib.accept_greedy(p, inp["draft_greedy"])
    assert np.array_equal(n.cpu().numpy(), n_ref) and np.array_equal(t.cpu().numpy(), t_ref), (B, D, V)
    n, t = sv.accept_sample(to_dev(p), to_dev(inp["q"]) if D else None, to_dev(inp["draft"]) if D else None,
                            to_dev(inp["u_acc"]) if D else None, to_dev(inp["u_res"]))
    torch.cuda.synchronize()
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, inp["q"], inp["draft"], inp["u_acc"], inp["u_res"])
    bad = (n.cpu().numpy() != n_ref) | (t.cpu().numpy() != t_ref)
    assert not (bad & (margin >= MARGIN)).any(), (B, D, V)
    tally(bad)


@pytest.mark.parametrize("seed", range(12))
def test_random_tree_attention(sv, oracle_lib, seed):
    import torch
    rng = np.random.default_rng(7000 + seed)
    B, Hkv, G, d, D, lens, page = attention_shape(rng)
    kind = str(rng.choice(["random", "star", "wide", "chain"]))
    inp = synth.attention_inputs(8000 + seed, B, Hkv, G, d, D, lens, page_size=page)
    parent = synth.tree_parents(9000 + seed, B, 1 + D, kind)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sv.verify_tree_attention(bits_dev(inp.q), bits_dev(inp.k_pages), bits_dev(inp.v_pages),
                                   to_dev(inp.block_table), to_dev(inp.kv_len), to_dev(parent), D, Hkv, G,
                                   dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, _ = oracle_lib.tree_attention(inp.q, inp.k_pages, inp.v_pages, inp.block_table, inp.kv_len, parent,
                                       D, Hkv, G, d, page)
    err = out.cpu().numpy().astype(np.float64) - ref
    assert np.abs(err).max() <= 2e-2, (B, Hkv, G, d, D, page, kind)
    assert np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref), (B, Hkv, G, d, D, page, kind)


@pytest.mark.parametrize("seed", range(8))
def test_random_tree_greedy(sv, oracle_lib, seed):
    import torch
    rng = np.random.default_rng(10000 + seed)
    B = int(rng.integers(1, 40))
    D = int(rng.integers(1, 16))
    V = int(rng.choice([7, 1000, 4099, 32768, 65536]))
    kind = str(rng.choice(["random", "star", "wide", "chain"]))
    p = synth.accept_inputs(11000 + seed, B, D, V, mode="greedy")["p"]
    parent = synth.tree_parents(12000 + seed, B, 1 + D, kind)
    am = np.argmax(p, axis=2)
    tokens = rng.integers(0, V, size=(B, 1 + D)).astype(np.int32)
    hit = rng.random((B, 1 + D)) < 0.7
    for b in range(B):
        for k in range(1, 1 + D):
            if hit[b, k]:
                tokens[b, k] = am[b, parent[b, k]]
    n, t, path = sv.accept_tree_greedy(to_dev(p), to_dev(tokens), to_dev(parent))
    torch.cuda.synchronize()
    n_ref, t_ref, path_ref = oracle_lib.accept_tree_greedy(p, tokens, parent)
    assert np.array_equal(n.cpu().numpy(), n_ref), (B, D, V, kind)
    assert np.array_equal(t.cpu().numpy(), t_ref) and np.array_equal(path.cpu().numpy(), path_ref)


@pytest.mark.parametrize("seed", range(8))
def test_random_acceptance_from_logits(sv, oracle_lib, seed):
    import torch
    rng = np.random.default_rng(13000 + seed)
    B = int(rng.integers(1, 24))
    D = int(rng.integers(0, 10))
    V = int(rng.choice([3, 300, 4096, 9001, 32768, 65536]))
    T = float(rng.choice([0.5, 1.0, 1.7]))
    inp = synth.logits_inputs(14000 + seed, B, D, V, target_std=float(rng.uniform(1.0, 4.0)),
                              draft_noise=float(rng.uniform(0.2, 1.5)), temperature=T,
                              masked=int(rng.integers(0, 3)) * (V // 4))
    zp, zq, draft = inp["zp"], inp["zq"], inp["draft"]
    n, t = sv.accept_sample_logits(to_dev(zp), to_dev(zq) if D else None, to_dev(draft) if D else None, T, seed)
    torch.cuda.synchronize()
    p, q, u_acc, u_res = oracle_lib.logits_to_probs(zp, zq, T, seed)
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, q, draft, u_acc, u_res)
    bad = (n.cpu().numpy() != n_ref) | (t.cpu().numpy() != t_ref)
    assert not (bad & (margin >= MARGIN)).any(), (B, D, V, T)
    tally(bad)


def test_zz_boundary_disagreements_stay_below_the_cap():
    """Over every comparison of this module: at most 1e-4 of the sequences
    disagree with the oracle (each one at a draw within 1e-6 of a boundary)."""
    assert TALLY["disagree"] <= 1e-4 * max(TALLY["draws"], 1), TALLY
