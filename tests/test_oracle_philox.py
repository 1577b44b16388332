"""The oracle's counter-based noise.  Philox4x32-10 is pinned to the published
known-answer vectors (tests/golden/philox4x32_10_kat.json); the other checks
constrain the stream built on it by the algebra of its round, by output
statistics, and by the Gumbel-max law of the draws."""
import numpy as np

import pins
from oracle import sampler as osm


def _inverse_round(o, k0, k1):
    """Undo one round: lo0 = o3 and lo1 = o1 give c0, c2 through the
    multipliers' inverses mod 2^32; their products' high words give c1, c3."""
    inv0 = pow(osm.PHILOX_M[0], -1, 1 << 32)
    inv1 = pow(osm.PHILOX_M[1], -1, 1 << 32)
    out = []
    for o0, o1, o2, o3 in o.tolist():
        c0 = (o3 * inv0) & osm.MASK32
        c2 = (o1 * inv1) & osm.MASK32
        hi0 = (osm.PHILOX_M[0] * c0) >> 32
        hi1 = (osm.PHILOX_M[1] * c2) >> 32
        out.append([c0, o0 ^ hi1 ^ k0, c2, o2 ^ hi0 ^ k1])
    return np.array(out, dtype=np.uint64)


def test_known_answer_vectors():
    pins.check_philox_kat(osm.philox4x32_10)


def test_round_is_invertible():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 1 << 32, size=(500, 4), dtype=np.uint64)
    k0, k1 = 0x12345678, 0x9ABCDEF0
    assert np.array_equal(_inverse_round(osm.philox_round(c, k0, k1), k0, k1), c)


def test_words_look_uniform_and_streams_differ():
    from scipy.stats import chisquare
    w = osm.philox_words(np.arange(400_000), seed=42, offset=7)
    assert w.max() < (1 << 32)
    for shift in (24, 0):                              # top byte and low byte
        counts = np.bincount(((w >> np.uint64(shift)) & np.uint64(255)).astype(np.int64),
                             minlength=256)
        assert chisquare(counts).pvalue > 1e-4
    bits = np.unpackbits(w.astype(np.uint32).view(np.uint8))
    assert abs(bits.mean() - 0.5) < 2e-3
    assert not np.array_equal(w[:1000], osm.philox_words(np.arange(1000), seed=43, offset=7))
    assert not np.array_equal(w[:1000], osm.philox_words(np.arange(1000), seed=42, offset=8))
    assert np.array_equal(w[:1000], osm.philox_words(np.arange(1000), seed=42, offset=7))


def test_noise_is_exp1():
    E = osm.philox_exp_noise(40, 10_000, seed=3, offset=0)
    assert E.min() >= 0.0
    assert abs(E.mean() - 1.0) < 0.01 and abs(E.var() - 1.0) < 0.03
    # P(E > 2) = e^-2
    assert abs((E > 2.0).mean() - np.exp(-2.0)) < 0.004


def test_draws_follow_the_gumbel_law():
    from scipy.stats import chisquare
    row = np.array([1.0, -0.5, 2.0, 0.0, 0.3, -2.0, 1.2, 0.8])
    draws = 60_000
    ids, _ = osm.sample_philox(np.tile(row, (draws, 1)), np.full(draws, 0.8), seed=11, offset=5)
    counts = np.bincount(ids, minlength=row.size)
    p = np.exp(row / 0.8 - (row / 0.8).max())
    p /= p.sum()
    assert chisquare(counts, p * draws).pvalue > 1e-4


def test_unit_logits_pick_the_largest_word():
    # all logits equal: the token is the entry with the largest U, i.e. the
    # largest word >> 8 (lowest index on ties)
    B, V = 5, 333
    ids, _ = osm.sample_philox(np.zeros((B, V)), np.ones(B), seed=9, offset=1)
    w = osm.philox_words(np.arange(B * V), 9, 1).reshape(B, V) >> np.uint64(8)
    assert np.array_equal(ids, np.argmax(w, axis=1))
