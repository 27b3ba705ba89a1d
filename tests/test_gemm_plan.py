"""The verify GEMM's work split, enumerated on the host.

The kernels' roles walk the same tile and segment lists; these checks run
the library's own planner (through spec_verify_gemm_plan) and need no GPU.
Weight streaming (M <= 256): with split K over clusters of S (when the
tiles' clusters all fit), S equal k-ranges per tile in rank order, one CTA
each; with stream-K, coverage of every (tile, k-block) exactly once,
balance across CTAs, one owner per tile whose contributor range matches
the pieces, and the ordering that keeps the owners' waits free of cycles.
CTA pairs (M > 256): whole tiles of ragged width that cover every output
column once and spread evenly over the pairs.
"""
from collections import defaultdict

import numpy as np
import pytest

import speculative_decoding_verification_attention_gb300 as sv


@pytest.fixture(scope="module", autouse=True)
def built():
    """The planner runs inside the library: rebuild it if a source is newer."""
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()

SHAPES = [(8, 6144, 6144), (200, 6144, 6144), (256, 384, 640), (1, 128, 64), (100, 19456, 640),
          (64, 128, 6144), (256, 256, 4096), (33, 6272, 640), (128, 65536, 64), (64, 10240, 6144)]


def split_size(M, N, K, sms):
    """The cluster size C >= 2 when the plan splits K over clusters, else 0."""
    c = sv.gemm_plan_cluster(M, N, K, sms)
    return c if M <= 256 and c >= 2 else 0
PAIR_SHAPES = [(257, 6144, 6144), (384, 128, 6144), (512, 6144, 6144), (1024, 6144, 6144),
               (2048, 6144, 6144), (4096, 6144, 6144), (3000, 6272, 1024), (512, 256, 64),
               (65536, 128, 64), (300, 384, 128), (600, 19584, 512)]


@pytest.mark.parametrize("sms", [152, 148, 7, 1])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_stream_k_split(M, N, K, sms):
    seg = sv.gemm_plan(M, N, K, sms)
    if split_size(M, N, K, sms):
        pytest.skip("split K over clusters (test_split_k_clusters)")
    bn = 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
    tiles = N // 128
    max_units, max_contrib = sms, 4 if bn <= 64 else 2
    kblocks = K // 64
    assert (seg[:, 5] == bn).all()
    ctas = seg[:, 0]
    G = int(ctas.max()) + 1
    assert G <= max_units and set(ctas.tolist()) == set(range(G))
    assert (np.diff(ctas) >= 0).all()          # rows come in CTA order

    # every (tile, k-block) exactly once
    cover = np.zeros((tiles, kblocks), np.int32)
    for c, t, k0, k1, last, _ in seg:
        assert 0 <= t < tiles and 0 <= k0 < k1 <= kblocks
        cover[t, k0:k1] += 1
    assert (cover == 1).all()

    # balance: k-blocks per CTA differ by at most one tile's worth of rounding
    work = np.zeros(G, np.int64)
    for c, t, k0, k1, *_ in seg:
        work[c] += k1 - k0
    assert work.max() - work.min() <= 1

    by_tile = defaultdict(list)
    for i, (c, t, k0, k1, last, _) in enumerate(seg):
        by_tile[t].append((c, k0, k1, last, i))
    for t, pieces in by_tile.items():
        owners = [p for p in pieces if p[1] == 0]
        assert len(owners) == 1
        oc, _, ok1, last, _ = owners[0]
        others = sorted(p[0] for p in pieces if p[1] > 0)
        # the owner's contributor range is exactly the CTAs holding the rest
        assert others == list(range(oc + 1, last + 1))
        if ok1 == kblocks:
            assert last == oc
        assert last - oc <= max_contrib    # bounded number of partials to add
    for c in range(G):
        rows = [r for r in seg if r[0] == c]
        cuts = [i for i, r in enumerate(rows) if r[2] > 0]
        # one partial slot per CTA: at most one later piece, and it comes
        # before any segment in which this CTA waits for others
        assert len(cuts) <= 1
        waits = [i for i, r in enumerate(rows) if r[2] == 0 and r[4] > c]
        if cuts and waits:
            assert cuts[0] < min(waits)
        # an owned cut tile is the CTA's last segment (its stage ring is idle)
        assert all(i == len(rows) - 1 for i in waits)
        assert all(r[4] == -1 for r in rows if r[2] > 0)


@pytest.mark.parametrize("sms", [152, 148, 20])
@pytest.mark.parametrize("M,N,K", SHAPES + [(8, 2304, 1024), (100, 2688, 1024), (256, 2560, 1024),
                                           (64, 3712, 512), (256, 4608, 6144), (128, 9472, 640),
                                           (65, 6144, 6144), (200, 512, 128)])
def test_split_k_clusters(M, N, K, sms):
    """Split K over clusters of C CTAs: unit c is CTA c of the grid, rank
    c % C; within a cluster the CTAs that hold the same 128-row tile split
    its k-blocks into equal contiguous ranges in rank order (S single CTAs
    per tile, or S CTA pairs per 256-row pair tile, ranks 2p + h holding
    tile 2T + h); every (tile, k-block) is covered once; the first piece's
    row names the last CTA holding the same tile; and all clusters fit the
    estimate of num_sms / C resident clusters."""
    C = split_size(M, N, K, sms)
    if not C:
        return
    tiles, kblocks = N // 128, K // 64
    bn = 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
    seg = sv.gemm_plan(M, N, K, sms)
    G = len(seg)
    assert G % C == 0 and G // C <= sms // C
    assert (seg[:, 0] == np.arange(G)).all()
    assert (seg[:, 5] == bn).all()
    cover = np.zeros((tiles, kblocks), np.int32)
    for cl in range(G // C):
        rows = seg[cl * C:(cl + 1) * C]
        by_tile = defaultdict(list)
        for c, t, k0, k1, last, _ in rows:
            by_tile[int(t)].append((int(c), int(k0), int(k1), int(last)))
        S = len(next(iter(by_tile.values())))
        assert S >= 2 and all(len(v) == S for v in by_tile.values())
        assert len(by_tile) * S == C and len(by_tile) in (1, 2)
        if len(by_tile) == 2:
            assert M > 64 and N % 256 == 0        # CTA pairs: 256-row pair tiles
        for t, pieces in by_tile.items():
            pieces.sort()
            for i, (c, k0, k1, last) in enumerate(pieces):
                assert (k0, k1) == (i * kblocks // S, (i + 1) * kblocks // S) and k0 < k1
                assert last == (pieces[-1][0] if i == 0 else -1)
                cover[t, k0:k1] += 1
    assert (cover == 1).all()


def test_verify_layer_at_small_m_splits_over_clusters():
    """N = K = 6144, M <= 256, planned for 152 SMs (estimate: 152 / C
    clusters of C): 48 tiles of 128 w rows; M <= 64 in clusters of three
    single CTAs, 64 < M in clusters of three CTA pairs (the pair's MMAs
    share the x rows); 32 k-blocks per CTA, 144 CTAs either way."""
    for M, C in ((8, 3), (64, 3), (65, 6), (128, 6), (256, 6)):
        assert sv.gemm_plan_cluster(M, 6144, 6144, 152) == C
        seg = sv.gemm_plan(M, 6144, 6144, 152)
        assert len(seg) == 144 and ((seg[:, 3] - seg[:, 2]) == 32).all()
    assert sv.gemm_plan_cluster(512, 6144, 6144, 152) == 2     # CTA pairs, whole tiles
    assert sv.gemm_plan_cluster(64, 19456, 640, 152) == 1      # 152 tiles: stream-K


def pair_columns(seg, M):
    """(tile -> (row block, first column, width)) from the plan rows of a
    CTA-pair GEMM; tile t is row block t % tiles_m of column tile t // tiles_m."""
    tiles_m = -(-M // 256)
    width = {}
    for c, t, k0, k1, last, w in seg:
        width[int(t) // tiles_m] = int(w)
    col0, acc = {}, 0
    for nt in sorted(width):
        col0[nt] = acc
        acc += width[nt]
    return tiles_m, width, col0, acc


@pytest.mark.parametrize("sms", [152, 148, 7, 2])
@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
def test_pair_tiles(M, N, K, sms):
    seg = sv.gemm_plan(M, N, K, sms)
    kblocks = K // 64
    assert ((seg[:, 2] == 0) & (seg[:, 3] == kblocks)).all()    # whole tiles
    assert (seg[:, 4] == seg[:, 0]).all()
    pairs = int(seg[:, 0].max()) + 1
    assert pairs <= max(1, sms // 2)
    tiles_m, width, col0, total = pair_columns(seg, M)
    tiles = tiles_m * len(width)
    # every tile exactly once; pair c takes tiles c, c + pairs, ...
    assert sorted(seg[:, 1].tolist()) == list(range(tiles))
    for c, t, *_ in seg:
        assert t % pairs == c
    per_pair = np.bincount(seg[:, 0], minlength=pairs)
    assert per_pair.max() - per_pair.min() <= 1
    # the column tiles cover N exactly; widths multiples of 32 within
    # [32, 256] that differ by at most 32, the wider ones first
    assert total == N
    ws = [width[nt] for nt in sorted(width)]
    assert all(w % 32 == 0 and 32 <= w <= 256 for w in ws)
    assert max(ws) - min(ws) <= 32
    assert ws == sorted(ws, reverse=True)
    # every (row block, column tile) is some tile's
    for c, t, k0, k1, last, w in seg:
        assert w == width[int(t) // tiles_m]


def test_verify_layer_at_512_rows_fills_every_pair():
    """N = K = 6144, M = 512, 76 resident pairs: 38 column tiles (2 of 192
    and 36 of 160 columns) x 2 row blocks = one whole tile per pair."""
    seg = sv.gemm_plan(512, 6144, 6144, 152)
    assert len(seg) == 76 and int(seg[:, 0].max()) + 1 == 76
    assert sorted(np.unique(seg[:, 5], return_counts=True)[1].tolist()) == [4, 72]
    assert set(seg[:, 5].tolist()) == {160, 192}


def test_weight_streaming_cuts_each_tile_in_thirds_at_small_m():
    """M = 8, N = K = 6144: the 48 w tiles of 128 rows are cut into three
    equal k-ranges of 32 k-blocks, one per CTA (144 of the 152 SMs stream
    weights), as clusters of three."""
    seg = sv.gemm_plan(8, 6144, 6144, 152)
    assert int(seg[:, 0].max()) + 1 == 144
    assert (seg[:, 5] == 32).all()
    assert ((seg[:, 3] - seg[:, 2]) == 32).all()
    assert sorted(np.bincount(seg[:, 1]).tolist()) == [3] * 48


def test_rejects_bad_arguments():
    lib = sv.library()
    assert lib.spec_verify_gemm_plan(512, 100, 64, 152, None, 0) == -1
    assert lib.spec_verify_gemm_plan(512, 128, 60, 152, None, 0) == -1
    assert lib.spec_verify_gemm_plan(512, 128, 64, 0, None, 0) == -1
    assert lib.spec_verify_gemm_plan(512, 128, 64, 152, None, 4) == -1
    assert lib.spec_verify_gemm_plan_cluster(512, 100, 64, 152) == -1
    assert lib.spec_verify_gemm_plan_cluster(512, 128, 64, 0) == -1


def test_small_m_few_tiles_are_cut():
    """M = 200, 3 tiles of 128 w rows over K = 6144 for 152 SMs: the k-blocks
    are split so that every CTA streams weights."""
    seg = sv.gemm_plan(200, 384, 6144, 152)
    assert int(seg[:, 0].max()) + 1 > 3
    assert ((seg[:, 2] > 0) | (seg[:, 3] < 96)).any()
