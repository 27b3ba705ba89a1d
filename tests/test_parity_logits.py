"""GPU parity of spec_accept_sample_logits against the oracle.

The oracle takes the fp64 softmax of logits / T rounded to fp32 (the fp32
probability rows of the probability form) and runs the fp64 acceptance on
them with its own Philox uniforms.  n_accepted and token are compared
element by element: bit-exact, except a draw whose oracle margin is below
1e-6; such disagreements are tallied over the whole module and must stay
at most 1e-4 of the sequences compared (the last test checks the tally).
The row statistics the library leaves in the workspace are checked too:
the maxima bit for bit, the fast fp32 sums Zf within their rounding bound
of the oracle's fp64 sums.  The device Philox is checked bit for bit
through uniform rows of 2^24 entries, where the drawn token is the 24-bit
integer of the uniform itself.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

MARGIN = 1e-6
# Zf sums at most 64 hardware exponentials per thread, then 8 + 3 tree
# levels, in fp32: relative error below (64 + 11) 2^-24 plus the
# exponential's own ~2^-22
ZF_REL = 1e-5
TALLY = {"draws": 0, "disagree": 0}


@pytest.fixture(scope="module")
def sv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(sv, zp, zq, draft, T, seed, dev_status=None, workspace=None):
    import torch
    B, D1, V = zp.shape
    D = D1 - 1
    if workspace is None:
        workspace = torch.empty(sv.accept_sample_logits_workspace_size(B, D, V), dtype=torch.uint8,
                                device="cuda")
    n, t = sv.accept_sample_logits(to_dev(zp), to_dev(zq) if D else None, to_dev(draft) if D else None,
                                   T, seed, workspace=workspace, dev_status=dev_status)
    torch.cuda.synchronize()
    rows = B * (2 * D + 1)
    stats = workspace[:rows * 8].cpu().numpy().view(np.float32).reshape(B, 2 * D + 1, 2)
    return n.cpu().numpy(), t.cpu().numpy(), stats


def compare(n, t, n_ref, t_ref, margin):
    """Bit-exact except draws within MARGIN of a decision boundary; tallied."""
    bad = (n != n_ref) | (t != t_ref)
    assert not (bad & (margin >= MARGIN)).any(), np.nonzero(bad & (margin >= MARGIN))
    TALLY["draws"] += len(n)
    TALLY["disagree"] += int(bad.sum())
    return bad


def check_stats(stats, m_ref, Z_ref):
    assert np.array_equal(stats[..., 0].view(np.uint32), m_ref.view(np.uint32))
    finite = np.isfinite(Z_ref)
    assert np.array_equal(np.isfinite(stats[..., 1]), finite)
    if finite.any():
        assert np.abs(stats[..., 1][finite] / Z_ref[finite] - 1).max() <= ZF_REL


def check(sv, oracle_lib, inp, T=None, seed=None):
    zp, zq, draft = inp["zp"], inp["zq"], inp["draft"]
    T = inp["temperature"] if T is None else T
    seed = inp["seed"] if seed is None else seed
    n, t, stats = run(sv, zp, zq, draft, T, seed)
    check_stats(stats, *oracle_lib.logits_row_stats(zp, zq, T))
    p, q, u_acc, u_res = oracle_lib.logits_to_probs(zp, zq, T, seed)
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, q, draft, u_acc, u_res)
    compare(n, t, n_ref, t_ref, margin)
    D = zp.shape[1] - 1
    assert n.min() >= 0 and n.max() <= D
    return n, t


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_small_step(sv, oracle_lib, seed):
    """One sequence, D = 3, V = 1000: target logits N(0, 2^2), draft logits
    the target's plus N(0, 0.5^2)."""
    inp = synth.logits_inputs(seed, 1, 3, 1000, target_std=2.0, draft_noise=0.5)
    check(sv, oracle_lib, inp)


@pytest.mark.parametrize("V", [1, 3, 7, 1001, 2048, 4099, 8192, 32768, 50257, 131072])
@pytest.mark.parametrize("D", [0, 1, 5])
def test_vocab_shapes_and_cluster_paths(sv, oracle_lib, V, D):
    """V from 1 to 131072 covers one- to eight-CTA clusters per row, bulk
    copies (V % 4 == 0) and plain loads (ragged V)."""
    inp = synth.logits_inputs(V + 7 * D, 12, D, V, target_std=3.0, draft_noise=0.7)
    check(sv, oracle_lib, inp)


@pytest.mark.parametrize("T", [0.25, 0.7, 1.0, 1.6])
def test_temperatures(sv, oracle_lib, T):
    inp = synth.logits_inputs(50 + int(T * 10), 16, 4, 20000, target_std=3.0, draft_noise=0.8,
                              temperature=T)
    check(sv, oracle_lib, inp)


def test_masked_vocabulary(sv, oracle_lib):
    """-inf logits (a masked vocabulary) have probability 0 on both sides."""
    inp = synth.logits_inputs(61, 10, 3, 32768, masked=5000)
    n, t = check(sv, oracle_lib, inp)
    for b in range(10):
        assert np.isfinite(inp["zp"][b, n[b], t[b]])


def test_max_draft_length(sv, oracle_lib):
    inp = synth.logits_inputs(62, 3, 63, 3000, draft_noise=0.05)
    check(sv, oracle_lib, inp)


def test_identical_models_accept_everything(sv, oracle_lib):
    inp = synth.logits_inputs(63, 32, 7, 8192)
    inp["zq"] = np.ascontiguousarray(inp["zp"][:, :7, :])
    n, _ = check(sv, oracle_lib, inp)
    assert (n == 7).all()


def test_device_philox_bit_exact(sv):
    """Equal logits over V = 2^24 make every target row uniform (p = 2^-24
    exactly), so with D = 0 the drawn token is u_res * 2^24 = the top 24
    bits of Philox word 0 for counter (b, 0, 1, 0)."""
    B, V = 4, 1 << 24
    zp = np.zeros((B, 1, V), np.float32)
    zq = np.zeros((B, 0, V), np.float32)
    draft = np.zeros((B, 0), np.int32)
    for seed in (0, 12345, 0xDEADBEEFCAFEF00D):
        n, t, _ = run(sv, zp, zq, draft, 1.0, seed)
        _, u_res = synth.acceptance_uniforms(seed, B, 0)
        assert (n == 0).all()
        assert np.array_equal(t.astype(np.int64), (u_res.astype(np.float64) * 2 ** 24).astype(np.int64))


def test_device_accept_uniforms(sv):
    """A draft with q = 1 and p = 2^-j is accepted iff u_acc < 2^-j: over
    many sequences and j in 0..4 the acceptance pattern reads the leading
    bits of every device uniform, which must match the published Philox
    (synth's independent implementation)."""
    B, D, V = 512, 1, 16
    rng = np.random.default_rng(0)
    j = rng.integers(0, 5, B)
    zp = np.full((B, 2, V), -np.inf, np.float32)
    zq = np.full((B, 1, V), -np.inf, np.float32)
    zq[:, 0, 0] = 0.0            # q(0) = 1: the only finite draft logit
    zp[:, 1, :] = 0.0            # the bonus row is uniform
    for b in range(B):
        zp[b, 0, :1 << j[b]] = 0.0   # 2^j equal target logits: p(0) = 2^-j exactly
    draft = np.zeros((B, 1), np.int32)
    seed = 77
    n, _, _ = run(sv, zp, zq, draft, 1.0, seed)
    u_acc, _ = synth.acceptance_uniforms(seed, B, 1)
    expect = (u_acc[:, 0].astype(np.float64) < 2.0 ** -j.astype(np.float64)).astype(np.int32)
    assert np.array_equal(n, expect)


def test_nonfinite_rows_are_flagged(sv, oracle_lib):
    import torch
    inp = synth.logits_inputs(64, 6, 2, 4096)
    zp, zq = inp["zp"].copy(), inp["zq"].copy()
    zp[1, 0, 17] = np.nan
    zq[3, 1, :] = -np.inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, stats = run(sv, zp, zq, inp["draft"], 1.0, 5, dev_status=st)
    assert int(st.item()) & sv.DEV_STATUS_BITS["LOGITS"]
    m_ref, Z_ref = oracle_lib.logits_row_stats(zp, zq, 1.0)
    check_stats(stats, m_ref, Z_ref)
    assert np.isinf(Z_ref[1, 0]) and np.isinf(Z_ref[3, 4])
    p, q, u_acc, u_res = oracle_lib.logits_to_probs(zp, zq, 1.0, 5)
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, q, inp["draft"], u_acc, u_res)
    compare(n, t, n_ref, t_ref, margin)


def test_workspace_reuse_and_graph_replay(sv, oracle_lib):
    """One workspace for calls of several shapes, then the call captured in a
    CUDA graph and replayed: every result matches the oracle."""
    import torch
    B, V = 24, 20000
    ws = torch.empty(sv.accept_sample_logits_workspace_size(B, 6, V), dtype=torch.uint8, device="cuda")
    for seed, D in ((71, 3), (72, 0), (73, 6)):
        inp = synth.logits_inputs(seed, B, D, V)
        n, t, _ = run(sv, inp["zp"], inp["zq"], inp["draft"], 1.0, seed, workspace=ws)
        p, q, u_acc, u_res = oracle_lib.logits_to_probs(inp["zp"], inp["zq"], 1.0, seed)
        n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, q, inp["draft"], u_acc, u_res)
        compare(n, t, n_ref, t_ref, margin)
    inp = synth.logits_inputs(74, B, 5, V)
    zp, zq, dr = to_dev(inp["zp"]), to_dev(inp["zq"]), to_dev(inp["draft"])
    n_out = torch.empty(B, dtype=torch.int32, device="cuda")
    t_out = torch.empty(B, dtype=torch.int32, device="cuda")
    sv.accept_sample_logits(zp, zq, dr, 1.0, 74, n_accepted=n_out, token=t_out, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sv.accept_sample_logits(zp, zq, dr, 1.0, 74, n_accepted=n_out, token=t_out, workspace=ws)
    p, q, u_acc, u_res = oracle_lib.logits_to_probs(inp["zp"], inp["zq"], 1.0, 74)
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, q, inp["draft"], u_acc, u_res)
    for _ in range(3):
        n_out.fill_(-1)
        t_out.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        compare(n_out.cpu().numpy(), t_out.cpu().numpy(), n_ref, t_ref, margin)


def test_batched_full_size(sv, oracle_lib):
    """B = 256 sequences, D = 7, V = 131072, target logits N(0, 3^2), draft
    logits the target's plus N(0, 1.5^2), two seeds: maxima bit-exact, sums
    within their bound, decisions equal to the oracle's except at boundary
    draws."""
    for seed in (80, 81):
        inp = synth.logits_inputs(seed, 256, 7, 131072, target_std=3.0, draft_noise=1.5)
        n, _ = check(sv, oracle_lib, inp)
        assert 0 < n.mean() < 7


def test_zz_disagreements_stay_below_the_cap():
    """Over every comparison of this module: at most 1e-4 of the sequences
    disagree with the oracle (each of them at a boundary draw)."""
    assert TALLY["draws"] > 0
    assert TALLY["disagree"] <= 1e-4 * TALLY["draws"], TALLY
