"""The adaptive draft-length controller (spec_adaptive_*), on the host.

Pins are hand-computed from the rule: EMA_1 = mean AL of the first round,
EMA_r = beta * EMA_(r-1) + (1 - beta) * mean AL, AL = n_accepted + 1; the
next round uses the smallest tier >= EMA, else the largest.
"""
import numpy as np
import pytest

import speculative_decoding_verification_attention_gb300 as sv


@pytest.fixture(scope="module", autouse=True)
def built():
    """The planner runs inside the library: rebuild it if a source is newer."""
    from speculative_decoding_verification_attention_gb300 import _build
    _build.build()


def test_starts_at_the_largest_tier():
    c = sv.AdaptiveDraftLength((1, 3, 7), beta=0.5)
    assert c.draft_len == 7


def test_ema_and_tier_by_hand():
    c = sv.AdaptiveDraftLength((1, 3, 7), beta=0.5)
    # round 1: AL = [1, 1, 2, 4] -> mean 2.0 -> EMA 2.0 -> tier 3
    assert c.update([0, 0, 1, 3]) == 3 and c.ema == pytest.approx(2.0)
    # round 2: mean AL 4.0 -> EMA 0.5*2 + 0.5*4 = 3.0 -> tier 3 (3 >= 3)
    assert c.update([3, 3, 3, 3]) == 3 and c.ema == pytest.approx(3.0)
    # round 3: mean AL 4.0 -> EMA 3.5 -> tier 7
    assert c.update([3, 3, 3, 3]) == 7 and c.ema == pytest.approx(3.5)
    # rounds of nothing accepted pull it down: EMA 2.25, 1.625, 1.3125, ...
    ds = [c.update([0] * 8) for _ in range(8)]
    assert ds[0] == 3 and ds[-1] == 3
    # EMA reaches 1 only in the limit: D = 1 needs AL = 1 exactly
    c2 = sv.AdaptiveDraftLength((1, 3, 7), beta=0.0)
    assert c2.update([0, 0, 0]) == 1
    assert c2.update([1, 0, 0]) == 3


def test_saturated_tier_moves_up_and_idle_moves_down():
    c = sv.AdaptiveDraftLength((1, 3, 7), beta=0.0)
    assert c.update(np.full(16, 3)) == 7      # D=3 fully accepted: AL 4 > 3
    assert c.update(np.full(16, 1)) == 3      # AL 2 at D=7: back to 3
    assert c.update(np.zeros(16)) == 1


def test_empty_round_keeps_the_average():
    c = sv.AdaptiveDraftLength((2, 4), beta=0.9)
    c.update([1, 2])
    e = c.ema
    assert c.update([]) == c.draft_len and c.ema == e


@pytest.mark.parametrize("tiers,beta", [((3, 1), 0.5), ((1, 1), 0.5), ((1, 3), 1.0), ((1, 3), -0.1),
                                        ((1, 64), 0.5), (tuple(range(9)), 0.5), ((), 0.5)])
def test_rejects_bad_configurations(tiers, beta):
    with pytest.raises(Exception):
        sv.AdaptiveDraftLength(tiers, beta)
