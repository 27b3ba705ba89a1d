"""GPU parity of spec_verify_gemm against the fp64 oracle.

Bar: relative L2 error <= 5e-3 over the compared entries (bf16 output
rounding alone gives ~1e-3), plus an elementwise bound of 2^-7 |y| + 1e-3.
Small shapes are compared in full; the verify shapes (N = K = 6144,
M = B(1+D) from 8 to 4096) on a seeded sample of entries that covers every
128-row / 128-column tile edge and every edge of the ragged column tiles of
the CTA-pair path, plus a full-tensor comparison with torch's
fp32-accumulating matmul as a secondary property check.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3


@pytest.fixture(scope="module")
def sv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()
    import speculative_decoding_verification_attention_gb300 as m
    m.library()
    return m


def bits_to_dev(bits):
    import torch
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def run(sv, x, w):
    import torch
    y = sv.verify_gemm(bits_to_dev(x), bits_to_dev(w))
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64), y


def check(y, ref):
    err = y - ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2, rel
    assert (np.abs(err) <= 2 ** -7 * np.abs(ref) + 1e-3).all(), np.abs(err).max()
    return rel


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (8, 256, 512), (31, 384, 640), (64, 128, 1024),
                                   (100, 256, 256), (128, 512, 128), (200, 128, 192),
                                   (256, 256, 512), (257, 256, 256), (300, 512, 320),
                                   (512, 384, 256)])
def test_full_compare_small(sv, oracle_lib, M, N, K):
    x, w = synth.gemm_inputs(M + N + K, M, N, K)
    y, _ = run(sv, x, w)
    check(y, oracle_lib.gemm(x, w))


@pytest.mark.parametrize("M,N,K", [(1, 6144, 512), (8, 6144, 640), (32, 6144, 64), (33, 6272, 640),
                                   (64, 6144, 576), (128, 6272, 512), (17, 384, 192), (100, 19456, 640),
                                   (5, 19584, 512), (24, 6272, 6144)])
def test_weight_streaming_full_compare(sv, oracle_lib, M, N, K):
    """Small-M weight streaming over the full width of the verify layer
    (and widths around it): every output against the oracle, so every
    128-row w tile, including the fp32 partials of tiles whose k-blocks are
    cut between CTAs, of which only the columns that hold rows of x are
    published and added."""
    x, w = synth.gemm_inputs(M * 7 + N + K, M, N, K)
    y, _ = run(sv, x, w)
    check(y, oracle_lib.gemm(x, w))


def pair_column_edges(sv, M, N, K):
    """First and last column of every column tile of the CTA-pair plan."""
    if M <= 256:
        return np.zeros(0, np.int64)
    seg = sv.gemm_plan(M, N, K, 152)
    tiles_m = -(-M // 256)
    width = {int(t) // tiles_m: int(w) for _, t, _, _, _, w in seg}
    edges, acc = [], 0
    for nt in sorted(width):
        edges += [acc, acc + width[nt] - 1]
        acc += width[nt]
    return np.asarray(edges, np.int64)


def sample_entries(rng, M, N, n=3000, col_edges=()):
    m = rng.integers(0, M, n)
    c = rng.integers(0, N, n)
    edges_m = np.unique(np.clip(np.concatenate([[0, M - 1], np.arange(127, M, 128),
                                                np.arange(128, M, 128)]), 0, M - 1))
    edges_n = np.unique(np.clip(np.concatenate([[0, N - 1], np.arange(127, N, 128),
                                                np.arange(128, N, 128)]), 0, N - 1))
    em, en = np.meshgrid(edges_m[:64], edges_n[:64])
    m = np.concatenate([m, em.ravel()])
    c = np.concatenate([c, en.ravel()])
    if len(col_edges):
        # every ragged column-tile edge, on rows at the row-block edges
        em, en = np.meshgrid(edges_m[:16], np.asarray(col_edges))
        m = np.concatenate([m, em.ravel()])
        c = np.concatenate([c, en.ravel()])
    return np.stack([m, c], axis=1).astype(np.int32)


@pytest.mark.parametrize("M", [8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 56, 120, 504])
def test_verify_shapes_sampled(sv, oracle_lib, M):
    import torch
    N = K = 6144
    x, w = synth.gemm_inputs(1000 + M, M, N, K)
    y, ydev = run(sv, x, w)
    rng = np.random.default_rng(M)
    s = sample_entries(rng, M, N, col_edges=pair_column_edges(sv, M, N, K))
    ref = oracle_lib.gemm(x, w, samples=s)
    check(y[s[:, 0], s[:, 1]], ref)
    # whole-tensor property: agrees with an fp32-accumulating library matmul
    yt = (bits_to_dev(x).float() @ bits_to_dev(w).float().T)
    rel = (ydev.float() - yt).norm() / yt.norm()
    assert float(rel) < REL_L2


def test_split_k_status_clear_and_repeatable(sv):
    """Split K over clusters of 3 (M = 128, N = K = 6144): no status bit, and
    a second call gives the same bits (the pieces are added in k order)."""
    import torch
    x, w = synth.gemm_inputs(23, 128, 6144, 6144)
    xd, wd = bits_to_dev(x), bits_to_dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = sv.verify_gemm(xd, wd, dev_status=st).clone()
    b = sv.verify_gemm(xd, wd, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(a, b)


def test_two_calls_in_a_row_agree(sv):
    x, w = synth.gemm_inputs(5, 64, 768, 6144)
    a, _ = run(sv, x, w)
    b, _ = run(sv, x, w)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M,N,K", [(200, 128, 6144), (256, 256, 4096), (64, 384, 6144), (8, 2304, 1024),
                                   (100, 2688, 1024), (256, 2560, 1024), (64, 3712, 512), (31, 4608, 1024),
                                   (256, 6144, 1024), (128, 9472, 640), (1, 1024, 128)])
def test_split_k_clusters(sv, oracle_lib, M, N, K):
    """Weight streaming with each tile's k-blocks split over a cluster
    (sizes 2 to 8 across these shapes: few tiles and long K take 8, N = 6144
    takes 3, N = 9472 takes 2), the pieces exchanged through distributed
    shared memory and added in k order: every output against the oracle."""
    x, w = synth.gemm_inputs(7 * M + K + N, M, N, K)
    segs = sv.gemm_plan(M, N, K, 152)
    assert (segs[:, 2] > 0).any()          # tiles really are cut
    y, _ = run(sv, x, w)
    check(y, oracle_lib.gemm(x, w))


@pytest.mark.parametrize("M,N,K", [(100, 8192, 256), (129, 6144, 1024), (256, 6656, 512), (65, 6144, 640)])
def test_split_k_cta_pairs(sv, oracle_lib, M, N, K):
    """64 < M <= 256 with N a multiple of 256 and many tiles: split K over
    clusters of CTA pairs whose MMAs (M = 256 w rows) each read half of the
    padded x rows from each CTA of the pair; the pieces of the two k-halves
    added in shared memory.  Every output against the oracle."""
    x, w = synth.gemm_inputs(13 * M + K + N, M, N, K)
    y, _ = run(sv, x, w)
    check(y, oracle_lib.gemm(x, w))


@pytest.mark.parametrize("M,N,K", [(64, 10240, 6144), (200, 10240, 1024)])
def test_stream_k_wide_layers(sv, oracle_lib, M, N, K):
    """More 128-row tiles (80) than clusters of two can hold at once: the
    stream-K split, whose cut tiles add their fp32 partials through the
    workspace (checked against the oracle in full)."""
    assert sv.gemm_plan_cluster(M, N, K, 152) == 1
    x, w = synth.gemm_inputs(11 * M + K, M, N, K)
    y, _ = run(sv, x, w)
    check(y, oracle_lib.gemm(x, w))


@pytest.mark.parametrize("M,N,K", [(512, 6144, 256), (300, 6272, 128), (384, 128, 64), (1024, 768, 512),
                                   (257, 19584, 64), (768, 2304, 192), (2048, 6144, 64),
                                   (812, 1792, 128), (5072, 256, 64)])
def test_pair_tiles_full_compare(sv, oracle_lib, M, N, K):
    """CTA-pair path (M > 256): ragged column tiles of 32-column multiples,
    row blocks of 256 with a ragged last one, several tiles per pair; every
    output against the oracle."""
    x, w = synth.gemm_inputs(3 * M + N + K, M, N, K)
    assert sv.gemm_workspace_size(M, N, K) == 0
    y, _ = run(sv, x, w)
    check(y, oracle_lib.gemm(x, w))


def test_pair_status_clear_and_repeatable(sv):
    """The pair kernel reports nothing in the status word and gives
    bit-identical results call after call (whole tiles, fixed k order)."""
    import torch
    M, N, K = 512, 6144, 1024
    x, w = synth.gemm_inputs(17, M, N, K)
    xd, wd = bits_to_dev(x), bits_to_dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [sv.verify_gemm(xd, wd, dev_status=st).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_workspace_reused_and_left_zero(sv):
    """One zeroed workspace serves many weight-streaming calls: each call
    leaves the arrival counters zero again, and results are bit-identical
    (fixed summation order, whichever piece of a cut tile arrives last)."""
    import torch
    M, N, K = 64, 6144, 6144
    x, w = synth.gemm_inputs(11, M, N, K)
    xd, wd = bits_to_dev(x), bits_to_dev(w)
    ws = torch.zeros(sv.gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [sv.verify_gemm(xd, wd, workspace=ws, dev_status=st).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    counters = ws[:4096]                   # arrival counters of the cut tiles
    assert int(counters.count_nonzero()) == 0


def test_workspace_zeroed_again_after_stale_counters(sv, oracle_lib):
    """A call that stops on its bounded wait may leave arrival counters
    non-zero; the contract is to zero the workspace again before the next
    call.  Stale counters are planted on the host side of that contract
    (the workspace filled with garbage), the workspace re-zeroed, and the
    next call must be exact."""
    import torch
    M, N, K = 32, 768, 6144
    x, w = synth.gemm_inputs(19, M, N, K)
    xd, wd = bits_to_dev(x), bits_to_dev(w)
    ws = torch.full((sv.gemm_workspace_size(M, N, K),), 7, dtype=torch.uint8, device="cuda")
    ws.zero_()
    y = sv.verify_gemm(xd, wd, workspace=ws)
    torch.cuda.synchronize()
    check(y.float().cpu().numpy().astype(np.float64), oracle_lib.gemm(x, w))
    assert int(ws[:4096].count_nonzero()) == 0


def test_graph_replay(sv, oracle_lib):
    """Captured once in a CUDA graph and replayed: every replay is right."""
    import torch
    M, N, K = 1024, 768, 6144
    x, w = synth.gemm_inputs(13, M, N, K)
    xd, wd = bits_to_dev(x), bits_to_dev(w)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(max(256, sv.gemm_workspace_size(M, N, K)), dtype=torch.uint8, device="cuda")
    sv.verify_gemm(xd, wd, y=y, workspace=ws)      # warm-up outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sv.verify_gemm(xd, wd, y=y, workspace=ws)
    ref = oracle_lib.gemm(x, w)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        check(y.float().cpu().numpy().astype(np.float64), ref)
