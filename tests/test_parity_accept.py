"""GPU parity of spec_accept_greedy / spec_accept_sample against the fp64
oracle, element by element (bit-exact on n_accepted and token).

A disagreement is tolerated only for a draw whose oracle margin (distance of
the uniform to the decision boundary) is below 1e-6, and the number of such
disagreements must stay below 1e-4 of the draws.  The kernel sums exactly
in fixed point, so in practice none occur.
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


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_greedy(sv, p, draft, dev_status=None):
    import torch
    n, t = sv.accept_greedy(to_dev(p), to_dev(draft), dev_status=dev_status)
    torch.cuda.synchronize()
    return n.cpu().numpy(), t.cpu().numpy()


def run_sample(sv, p, q, draft, u_acc, u_res, dev_status=None):
    import torch
    D = p.shape[1] - 1
    n, t = sv.accept_sample(to_dev(p), to_dev(q) if D else None, to_dev(draft) if D else None,
                            to_dev(u_acc) if D else None, to_dev(u_res), dev_status=dev_status)
    torch.cuda.synchronize()
    return n.cpu().numpy(), t.cpu().numpy()


def check_greedy(sv, oracle_lib, p, draft):
    n, t = run_greedy(sv, p, draft)
    n_ref, t_ref = oracle_lib.accept_greedy(p, draft)
    assert np.array_equal(n, n_ref)
    assert np.array_equal(t, t_ref)
    D = p.shape[1] - 1
    assert n.min() >= 0 and n.max() <= D          # AL = n + 1 in [1, 1 + D]
    return n


def check_sample(sv, oracle_lib, inp):
    p, q, draft, u_acc, u_res = inp["p"], inp["q"], inp["draft"], inp["u_acc"], inp["u_res"]
    n, t = run_sample(sv, p, q, draft, u_acc, u_res)
    n_ref, t_ref, margin, _ = oracle_lib.accept_sample(p, q, draft, u_acc, u_res)
    bad = (n != n_ref) | (t != t_ref)
    assert not (bad & (margin >= MARGIN)).any(), np.nonzero(bad & (margin >= MARGIN))
    tally(bad)
    D = p.shape[1] - 1
    assert n.min() >= 0 and n.max() <= D
    return n, t


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_step_both_modes(sv, oracle_lib, seed):
    inp = synth.accept_inputs(seed, 1, 3, 1000, target_std=2.0, draft_noise=0.5, mode="both")
    check_greedy(sv, oracle_lib, inp["p"], inp["draft_greedy"])
    check_sample(sv, oracle_lib, inp)


@pytest.mark.parametrize("V", [1, 3, 7, 1001, 2048, 4099, 8192, 32768, 40000, 50257, 200000])
@pytest.mark.parametrize("D", [0, 1, 5])
def test_vocab_shapes_and_cluster_paths(sv, oracle_lib, V, D):
    inp = synth.accept_inputs(V + D, 24, D, V, target_std=2.0, draft_noise=0.7, mode="both")
    check_greedy(sv, oracle_lib, inp["p"], inp["draft_greedy"])
    check_sample(sv, oracle_lib, inp)


def test_greedy_rows_without_16_byte_alignment(sv, oracle_lib):
    """p starting 4 bytes past a 16-byte boundary (V % 4 == 0): rows cannot
    be staged by bulk copies and take the register-load kernel; the results
    must not change."""
    import torch
    B, D, V = 24, 5, 32768
    inp = synth.accept_inputs(77, B, D, V, target_std=2.0, draft_noise=0.7, mode="both")
    p, draft = inp["p"], inp["draft_greedy"]
    flat = torch.empty(p.size + 1, dtype=torch.float32, device="cuda")
    flat[1:] = to_dev(p.reshape(-1))
    pd = flat[1:].view(B, D + 1, V)
    assert pd.data_ptr() % 16 == 4
    n, t = sv.accept_greedy(pd, to_dev(draft))
    torch.cuda.synchronize()
    n_ref, t_ref = oracle_lib.accept_greedy(p, draft)
    assert (n.cpu().numpy() == n_ref).all() and (t.cpu().numpy() == t_ref).all()


@pytest.fixture(scope="module")
def sigmas():
    return {a: synth.tune_sigma_for_alpha(a, 131072, rows=16, target_std=3.0)[0]
            for a in (0.4, 0.6, 0.8)}


@pytest.mark.parametrize("alpha", [0.4, 0.6, 0.8])
def test_batched_acceptance_full_size(sv, oracle_lib, sigmas, alpha):
    """B=256 sequences, D=7, V=131072, target logits N(0, 3^2)."""
    inp = synth.accept_inputs(40 + int(alpha * 10), 256, 7, 131072, target_std=3.0,
                              draft_noise=sigmas[alpha], mode="both")
    ng = check_greedy(sv, oracle_lib, inp["p"], inp["draft_greedy"])
    ns, _ = check_sample(sv, oracle_lib, inp)
    # the stochastic rule accepts at about the tuned rate
    assert abs(ns.mean() - (alpha - alpha ** 8) / (1 - alpha)) < 1.0
    assert ng.max() <= 7


def test_greedy_ties_across_cta_slices(sv, oracle_lib):
    V, D = 131072, 2
    p = np.full((3, D + 1, V), 1e-6, np.float32)
    p[0, :, 100000] = 0.5
    p[0, :, 5] = 0.5           # tie: lowest index wins
    p[1, :, 77777] = 0.25
    p[1, :, 131071] = 0.25
    p[2, :, 0] = 0.125
    p[2, :, 65536] = 0.125
    draft = np.array([[5, 5], [77777, 1], [3, 0]], np.int32)
    n = check_greedy(sv, oracle_lib, p, draft)
    assert list(n) == [2, 1, 0]


def test_zero_residual_fallback_and_flag(sv, oracle_lib):
    import torch
    V = 4096
    p = np.full((2, 2, V), 1.0 / V, np.float32)
    q = np.full((2, 1, V), 1.0 / V, np.float32)
    p[:, 0, 7] = 0.0                     # p <= q everywhere: Z = 0 after a rejection
    draft = np.array([[7], [7]], np.int32)
    u_acc = np.array([[0.5], [0.0]], np.float32)
    u_res = np.array([0.3, 0.9], np.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t = run_sample(sv, p, q, draft, u_acc, u_res, dev_status=st)
    n_ref, t_ref, _, fb = oracle_lib.accept_sample(p, q, draft, u_acc, u_res)
    assert fb.all()
    assert np.array_equal(n, n_ref) and np.array_equal(t, t_ref)
    assert int(st.item()) & sv.DEV_STATUS_BITS["INFO_ZERO_RESIDUAL"]


def test_invalid_token_and_uniform_are_flagged(sv):
    import torch
    V, D = 1000, 2
    inp = synth.accept_inputs(9, 4, D, V, mode="sample")
    draft = inp["draft"].copy()
    draft[1, 0] = V + 5
    u_res = inp["u_res"].copy()
    u_res[2] = 1.5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t = run_sample(sv, inp["p"], inp["q"], draft, inp["u_acc"], u_res, dev_status=st)
    bits = int(st.item())
    assert bits & sv.DEV_STATUS_BITS["TOKEN_ID"] and bits & sv.DEV_STATUS_BITS["UNIFORM"]
    assert n[1] == 0 and 0 <= t.min() and t.max() < V


def test_rows_that_are_not_probabilities_are_flagged(sv):
    """The values a sequence draws from must lie in [0, 2) and sum below 8
    (its exact 2^-61 masses fit in 64 bits); a NaN, a negative entry, an
    entry of 2 or more or a row summing past 8 sets the PROB bit, while a
    valid row, -0 entries included, does not."""
    import torch
    B, D, V = 6, 1, 3000
    rng = np.random.default_rng(5)
    q = rng.random((B, D, V)).astype(np.float32)
    q /= q.sum(axis=-1, keepdims=True)
    p = np.empty((B, D + 1, V), np.float32)
    p[:, :D] = q                   # p = q: every draft accepted, the draw reads p[b][D]
    p[:, D] = q[:, 0]
    p[1, D, 17] = np.nan
    p[2, D, V - 1] = -0.25
    p[3, D, 100] = 2.5
    p[4, D, :] = 0.9               # sums to 2700
    p[5, D, :] = 0.01              # every 512-element group below 8, the row at 30
    p[0, D, :40] = -0.0            # -0 is a zero probability
    draft = np.zeros((B, D), np.int32)
    u_acc = np.full((B, D), 0.5, np.float32)
    u_res = np.full(B, 0.5, np.float32)
    for rows, flagged in (([0], False), ([0, 1], True), ([2], True), ([3, 0], True), ([4], True), ([5], True)):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        n, t = run_sample(sv, p[rows], q[rows], draft[rows], u_acc[rows], u_res[rows], dev_status=st)
        assert bool(int(st.item()) & sv.DEV_STATUS_BITS["PROB"]) == flagged, rows
        assert (n == D).all() and 0 <= t.min() and t.max() < V


def test_repeat_calls_are_identical(sv, oracle_lib):
    inp = synth.accept_inputs(3, 64, 4, 20000, mode="both")
    a = run_sample(sv, inp["p"], inp["q"], inp["draft"], inp["u_acc"], inp["u_res"])
    b = run_sample(sv, inp["p"], inp["q"], inp["draft"], inp["u_acc"], inp["u_res"])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_one_workspace_serves_many_calls(sv, oracle_lib):
    """One workspace is reused by calls with different draft lengths (so
    different rows are streamed): every result is exact."""
    import torch
    B, V = 48, 20000
    ws = torch.empty(sv.accept_sample_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    for seed, D in ((21, 3), (22, 0), (23, 6)):
        inp = synth.accept_inputs(seed, B, D, V, mode="sample")
        n, t = sv.accept_sample(to_dev(inp["p"]), to_dev(inp["q"]) if D else None,
                                to_dev(inp["draft"]) if D else None,
                                to_dev(inp["u_acc"]) if D else None, to_dev(inp["u_res"]), workspace=ws)
        torch.cuda.synchronize()
        n_ref, t_ref, margin, _ = oracle_lib.accept_sample(inp["p"], inp["q"], inp["draft"], inp["u_acc"],
                                                           inp["u_res"])
        bad = (n.cpu().numpy() != n_ref) | (t.cpu().numpy() != t_ref)
        assert not (bad & (margin >= MARGIN)).any()
        tally(bad)


def test_greedy_calls_with_changing_shapes(sv, oracle_lib):
    """Back-to-back calls with different draft lengths on one stream: every
    result is exact (the per-row exchange state starts fresh each call)."""
    B, V = 40, 30000
    for seed, D in ((31, 7), (32, 0), (33, 3), (34, 7)):
        inp = synth.accept_inputs(seed, B, D, V, mode="greedy")
        check_greedy(sv, oracle_lib, inp["p"], inp["draft"])


def test_greedy_deep_rows_many_sequences(sv, oracle_lib):
    """Drafts equal to the target argmax for most positions: sequences run
    through many rows, so later rows wait on earlier decisions."""
    B, D, V = 300, 7, 9000
    inp = synth.accept_inputs(41, B, D, V, mode="greedy")
    p = inp["p"]
    draft = np.argmax(p[:, :D, :], axis=2).astype(np.int32)
    rng = np.random.default_rng(5)
    flip = rng.random((B, D)) < 0.1
    draft[flip] = (draft[flip] + 1) % V
    n = check_greedy(sv, oracle_lib, p, draft)
    assert (n == D).sum() > 10


def test_zz_boundary_disagreements_stay_below_the_cap():
    """Over every comparison of this module: at most 1e-4 of the sequences
    disagree with the oracle (each one at a draw within 1e-6 of a boundary)."""
    assert TALLY["disagree"] <= 1e-4 * max(TALLY["draws"], 1), TALLY
