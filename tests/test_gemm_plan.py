"""The tiled verify GEMM's stream-K split, enumerated on the host.

The kernel's three roles walk the same segment list; these checks run the
library's own walker (through spec_verify_gemm_plan) and need no GPU:
coverage of every (tile, k-block) exactly once, balance across CTAs, one
owner per tile whose contributor range matches the pieces, and the
ordering that keeps the owners' waits free of cycles.
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

SHAPES = [(8, 6144, 6144), (200, 6144, 6144), (256, 384, 640), (1, 128, 64), (257, 6144, 6144), (384, 128, 6144), (512, 6144, 6144), (1024, 6144, 6144),
          (2048, 6144, 6144), (4096, 6144, 6144), (3000, 6272, 1024), (512, 256, 64),
          (65536, 128, 64), (300, 384, 128)]


@pytest.mark.parametrize("sms", [152, 148, 7, 1])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_stream_k_split(M, N, K, sms):
    seg = sv.gemm_plan(M, N, K, sms)
    swap = M <= 256
    if swap:        # 128-row w tiles; x rows padded to the MMA N
        bn = 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
        tiles = N // 128
        max_units, max_contrib = sms, 4 if bn <= 64 else 2
    else:           # 256-row pair tiles
        bn = 256 if N % 256 == 0 else 128
        tiles = -(-(-(-M // 128)) // 2) * (N // bn)
        max_units, max_contrib = max(1, sms // 2), 2
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
    first_sk = {}
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


def test_weight_streaming_cuts_each_tile_in_thirds_at_small_m():
    """M = 8, N = K = 6144: the 48 w tiles of 128 rows are cut into three
    equal k-ranges of 32 k-blocks, one per CTA (144 of the 152 SMs stream
    weights)."""
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


@pytest.mark.parametrize("M", [384, 512, 640, 768])
def test_half_to_full_wave_takes_whole_tiles(M):
    """N = K = 6144 with 76 resident CTA pairs: 48 or 72 pair tiles fill at
    least half of the pairs, so every pair takes one whole tile and no tile
    is cut (nothing to add up through the workspace)."""
    N = K = 6144
    seg = sv.gemm_plan(M, N, K, 152)
    tiles = -(-(-(-M // 128)) // 2) * (N // 256)
    assert len(seg) == tiles
    assert sorted(seg[:, 1].tolist()) == list(range(tiles))
    assert (seg[:, 2] == 0).all() and (seg[:, 3] == K // 64).all()
    assert int(seg[:, 0].max()) + 1 == tiles


def test_less_than_half_a_wave_is_cut():
    """16 pair tiles for 76 pairs: the k-blocks are split so every pair works."""
    seg = sv.gemm_plan(512, 2048, 6144, 152)
    assert int(seg[:, 0].max()) + 1 > 16
    assert ((seg[:, 2] > 0) | (seg[:, 3] < 96)).any()
