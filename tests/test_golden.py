"""Fixtures of relations the source pages state (tests/golden/), checked on
the CPU: the attention cases the benchmark measures sit exactly on the
co-design blog's Guideline 2 draft length, and the large-group sweep
straddles the first 128-row tile boundary of its Figure 5."""
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load_guideline2():
    rows = []
    with open(os.path.join(HERE, "golden", "guideline2_draft_length.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(tuple(int(v) for v in line.split()))
    return np.array(rows)


def test_fixture_rows_fill_one_tile():
    g = load_guideline2()
    G, D, rows = g[:, 0], g[:, 1], g[:, 2]
    assert (D == 128 // G - 1).all()
    assert (G * (1 + D) == rows).all() and (rows == 128).all()


def bench_module():
    import sys
    root = os.path.dirname(HERE)
    if root not in sys.path:
        sys.path.insert(0, root)
    import bench
    return bench


def test_throughput_case_uses_guideline2_draft_length():
    g = {G: D for G, D, _ in load_guideline2()}
    c = bench_module().THROUGHPUT_CASE
    assert c["D"] == g[c["G"]] and c["G"] * (1 + c["D"]) == 128


def test_large_group_sweep_straddles_the_tile_boundary():
    g = {G: D for G, D, _ in load_guideline2()}
    c = bench_module().DSWEEP_CASE
    ds = list(c["Ds"])
    D0 = g[c["G"]]
    assert D0 in ds and D0 + 1 in ds          # last D of one tile, first D of two
    tiles = [-(-c["G"] * (1 + d) // 128) for d in ds]
    assert sorted(set(tiles)) == [1, 2, 4]    # one, two and four 128-row tiles
