"""The sampler oracle against closed forms and the Gumbel-max law."""
import numpy as np

import pins
from oracle import sampler as osm


def test_unit_noise_is_greedy():
    pins.check_unit_noise_is_greedy(osm.sample)


def test_gumbel_law_chi_square():
    pins.check_gumbel_law(osm.sample)


def test_lowest_index_tie():
    pins.check_lowest_index_tie(osm.sample)


def test_temperature_matters():
    pins.check_temperature_matters(osm.sample)


def test_two_statements_agree():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((64, 300)) * 3
    T = rng.uniform(0.2, 1.2, 64)
    E = rng.exponential(size=logits.shape)
    a, _ = osm.sample(logits, T, E)
    b, _ = osm.sample_key_form(logits, T, E)
    assert np.array_equal(a, b)


def test_bad_temperature_rows():
    logits = np.zeros((4, 5))
    logits[:, 3] = 1.0
    ids, bad = osm.sample(logits, np.array([0.0, -1.0, np.nan, 1.0]), np.ones((4, 5)))
    assert bad == [0, 1, 2] and ids.tolist() == [0, 0, 0, 3]


def test_noise_floor():
    # E = 0 is clamped to 1e-10, so that entry wins unless another key is larger
    logits = np.array([[0.0, 5.0]])
    ids, _ = osm.sample(logits, np.array([1.0]), np.array([[0.0, 1.0]]))
    assert ids.tolist() == [0]
