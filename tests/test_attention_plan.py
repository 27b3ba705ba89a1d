"""Host logic of the verify-attention KV split (the same code the kernels
run), checked through spec_verify_attention_plan: every key tile of every
(b, h) unit is processed exactly once, whole units go straight to the
output, partial segments use distinct slots (at most two per group), and
every group does (almost) the same number of tiles."""
import numpy as np
import pytest

import speculative_decoding_verification_attention_gb300 as sv


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()


CASES = [
    ([256], 3, 1, 152),
    ([32768] * 16, 15, 8, 152),
    ([131072] * 8, 15, 4, 38),
    (list(np.random.default_rng(0).integers(4096, 131073, 64)), 7, 8, 152),
    ([5, 1, 64, 65, 0, 129], 3, 3, 7),       # lengths < 1 + D are skipped
    ([10] * 3, 0, 2, 152),                   # fewer tiles than groups
]


@pytest.mark.parametrize("lens,D,Hkv,groups", CASES)
def test_plan_covers_each_tile_once(lens, D, Hkv, groups):
    kv = np.array(lens, np.int32)
    seg = sv.attention_plan(kv, D, Hkv, groups)
    kt = sv.ATTENTION_KEY_TILE
    nk = np.where(kv >= 1 + D, (kv.astype(np.int64) + kt - 1) // kt, 0)
    covered = {}
    per_group = {}
    slots = set()
    for g, b, h, t0, t1, slot in seg:
        assert 0 <= t0 < t1 <= nk[b]
        for t in range(t0, t1):
            assert (b, h, t) not in covered
            covered[(b, h, t)] = g
        per_group[g] = per_group.get(g, 0) + (t1 - t0)
        whole = (t0 == 0 and t1 == nk[b])
        assert (slot == -1) == whole
        if slot >= 0:
            assert slot in (2 * g, 2 * g + 1)
            assert slot not in slots
            slots.add(slot)
    assert len(covered) == int(nk.sum()) * Hkv
    counts = np.array(list(per_group.values()))
    assert counts.max() - counts.min() <= 1
    # segments of a group are consecutive in (b, h, tile) order
    for g in per_group:
        s = seg[seg[:, 0] == g]
        keys = [(b, h, t0) for _, b, h, t0, _, _ in s]
        assert keys == sorted(keys)


def test_plan_rejects_bad_arguments():
    lib = sv.library()
    assert lib.spec_verify_attention_plan(-1, None, 0, 1, 1, None, 0) == -1
    assert lib.spec_verify_attention_plan(1, None, 0, 1, 1, None, 0) == -1
