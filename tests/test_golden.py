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


def bench_source():
    with open(os.path.join(os.path.dirname(HERE), "bench.py")) as f:
        return f.read()


def test_throughput_case_uses_guideline2_draft_length():
    g = {G: D for G, D, _ in load_guideline2()}
    m = re.search(r'attention_case\("throughput B16 L32768 D(\d+)", 16, 8, (\d+), (\d+), 32768', bench_source())
    assert m, "throughput attention case not found"
    d_name, G, D = int(m.group(1)), int(m.group(2)), int(m.group(3))
    assert d_name == D == g[G]


def test_large_group_sweep_straddles_the_tile_boundary():
    g = {G: D for G, D, _ in load_guideline2()}
    m = re.search(r"for D in \(([0-9, ]+)\):\s*\n\s*attention_case\(f\"large-group B8 G32", bench_source())
    assert m, "large-group sweep not found"
    ds = [int(v) for v in m.group(1).split(",")]
    D0 = g[32]
    assert D0 in ds and D0 + 1 in ds          # last D of one tile, first D of two
    tiles = [-(-32 * (1 + d) // 128) for d in ds]
    assert sorted(set(tiles)) == [1, 2, 4]    # one, two and four 128-row tiles
