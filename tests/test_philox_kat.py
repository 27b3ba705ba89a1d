"""Known-answer pins for the Philox4x32-10 generator that draws the acceptance
uniforms (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11).

The input-generator module's Philox is checked against all three published
vectors word by word. The oracle's own C Philox is reachable only through the
uniforms it draws (word 0's top 24 bits at counter (b, i, stream, 0)), so it is
pinned at the one vector with that counter shape (all zeros, key 0), and it is
tied to the generator module on many other counters by the oracle tests.
"""
import os

import numpy as np

import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def load_kat():
    rows = []
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            w = [int(v, 16) for v in line.split()]
            assert len(w) == 10
            c0, c1, c2, c3, k0, k1 = w[:6]
            x = tuple(w[6:])
            rows.append(((c0, c1, c2, c3), k0 | (k1 << 32), x))
    return rows


def test_fixture_has_the_three_vectors():
    assert len(load_kat()) == 3


def test_generator_module_matches_known_answers():
    for counter, key, expected in load_kat():
        out = synth.philox4x32_10(*counter, key)
        assert tuple(int(w) for w in out) == expected


def test_generator_module_matches_known_answers_batched():
    # The same vectors evaluated as one broadcast call, so the vectorised
    # path (not only the scalar one) carries the pin.
    kat = [r for r in load_kat() if r[1] == 0]
    counters = np.array([r[0] for r in kat], dtype=np.uint64).T
    out = synth.philox4x32_10(*counters, 0)
    for j, (_, _, expected) in enumerate(kat):
        assert tuple(int(w[j]) for w in out) == expected


def test_uniform_is_top_24_bits_of_word_zero():
    (counter, key, expected), = [r for r in load_kat() if r[0] == (0, 0, 0, 0) and r[1] == 0]
    u = synth.philox_uniform(key, 0, 0, 0)
    assert float(u) == (expected[0] >> 8) * 2.0 ** -24


def test_oracle_uniform_matches_known_answer(oracle_lib):
    (_, _, expected), = [r for r in load_kat() if r[0] == (0, 0, 0, 0) and r[1] == 0]
    z = np.zeros((1, 2, 4), np.float32)
    _, _, u_acc, _ = oracle_lib.logits_to_probs(z, z[:, :1], 1.0, 0)
    assert float(u_acc[0, 0]) == (expected[0] >> 8) * 2.0 ** -24
