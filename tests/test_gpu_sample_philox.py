"""The in-kernel-noise sampler against the oracle's restatement of the same
Philox4x32-10 stream."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import sampler as osm
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("vocab", [4096, 4099])
@pytest.mark.parametrize("seed,offset", [(0, 0), (12345, 3), ((1 << 40) + 7, (1 << 33) + 1)])
def test_equal_logits_pick_the_largest_word_exactly(cuda, vocab, seed, offset):
    """With equal logits the key is -ln E = -ln(-ln U): the token is the entry
    with the largest U, i.e. the largest word >> 8, an integer decision the
    oracle makes exactly from its own Philox stream."""
    pkv = U.lib()
    B = 16
    ids = pkv.sample_philox(torch.zeros((B, vocab), device=cuda),
                            torch.ones(B, device=cuda), seed, offset).cpu().numpy()
    w = osm.philox_words(np.arange(B * vocab), seed, offset).reshape(B, vocab) >> np.uint64(8)
    assert np.array_equal(ids, np.argmax(w, axis=1))


@pytest.mark.parametrize("t_lo,t_hi", [(0.2, 1.2), (0.02, 0.2), (1.2, 4.0)])
def test_spiked_logits_full_vocab_rows(cuda, t_lo, t_hi):
    """Full 151936-entry rows of the step-8b sampler inputs at low, step-8b and
    high temperatures (the kernel computes the exact key only for entries that
    can still reach its running best, a share that depends on the spread)."""
    pkv = U.lib()
    B = 24
    g = torch.Generator().manual_seed(4)
    logits, temps, _ = W.sampler_inputs(B, 151936, 3.0, 4, t_lo, t_hi, g)
    ids = pkv.sample_philox(logits.to(cuda), temps.to(cuda), 99, 5).cpu().numpy()
    ref, bad = osm.sample_philox(logits.numpy(), temps.numpy(), 99, 5)
    E = osm.philox_exp_noise(B, 151936, 99, 5)
    _, keys = osm.sample_key_form(logits.numpy(), temps.numpy(), E)
    near = osm.near_ties(keys)
    assert not bad
    for r in range(B):
        assert ids[r] == ref[r] or (len(near[r]) > 1 and ids[r] in near[r])


def test_degenerate_rows(cuda):
    """Rows where only a few entries (or none) have a finite key: every key
    -inf gives the lowest index; one finite logit, or one +inf logit, wins; a
    row of NaN gives 0 and reports PKV_STATUS_NO_FINITE_KEY; a row of equal
    logits with one raised entry far above the rest picks that entry."""
    pkv = U.lib()
    V = 5003
    lg = torch.zeros(5, V)
    lg[0] = float("-inf")
    lg[1] = float("-inf")
    lg[1, 4321] = 0.0
    lg[2] = float("nan")
    lg[3] = float("-inf")
    lg[3, 17] = float("inf")
    lg[4] = 0.0
    lg[4, 2999] = 200.0
    temps = torch.tensor([1.0, 0.5, 1.0, 1.0, 0.7])
    st = pkv.new_status(cuda)
    ids = pkv.sample_philox(lg.to(cuda), temps.to(cuda), 5, 6, status=st).cpu().tolist()
    assert ids == [0, 4321, 0, 17, 2999]
    assert U.status_word(st) == pkv.STATUS["NO_FINITE_KEY"]


def test_draws_follow_the_gumbel_law(cuda):
    from scipy.stats import chisquare
    pkv = U.lib()
    row = torch.tensor([1.0, -0.5, 2.0, 0.0, 0.3, -2.0, 1.2, 0.8])
    draws = 40_000
    ids = pkv.sample_philox(row.repeat(draws, 1).to(cuda), torch.full((draws,), 0.8, device=cuda),
                            2024, 0).cpu().numpy()
    counts = np.bincount(ids, minlength=8)
    x = row.double().numpy() / 0.8
    p = np.exp(x - x.max())
    p /= p.sum()
    assert chisquare(counts, p * draws).pvalue > 1e-4


def test_bad_temperature_rows(cuda):
    pkv = U.lib()
    st = pkv.new_status(cuda)
    ids = pkv.sample_philox(torch.randn(3, 100, device=cuda),
                            torch.tensor([1.0, 0.0, float("inf")], device=cuda), 1, 1,
                            status=st).cpu().tolist()
    assert ids[1:] == [0, 0]
    assert U.status_word(st) == pkv.STATUS["BAD_TEMPERATURE"]


@pytest.mark.parametrize("vocab", [16, 13])
@pytest.mark.parametrize("seed,offset", [(7, 0), ((1 << 37) + 5, (1 << 35) + 2)])
def test_each_rows_noise_order_follows_the_oracle_words(cuda, vocab, seed, offset):
    """The whole noise of small rows, not only its largest entry: with equal
    logits the draw picks the entry with the largest U; masking each winner and
    drawing again V times gives the kernel's complete order of the row's U
    values, which must be the order of the oracle's Philox words (w >> 8).  A
    word taken from the wrong counter, lane or key shows as an out-of-order
    pair.  Entries whose float64 keys lie within 1e-5 of each other may come
    in either order (the kernel decides in float32)."""
    pkv = U.lib()
    B = 64
    logits = torch.zeros((B, vocab), device=cuda)
    temps = torch.ones(B, device=cuda)
    rows = torch.arange(B, device=cuda)
    order = np.zeros((B, vocab), dtype=np.int64)
    for k in range(vocab):
        ids = pkv.sample_philox(logits, temps, seed, offset)
        order[:, k] = ids.cpu().numpy()
        logits[rows, ids.long()] = -1.0e4            # masked: its key stays below -9000
    assert all(sorted(order[r].tolist()) == list(range(vocab)) for r in range(B))
    w = osm.philox_words(np.arange(B * vocab), seed, offset).reshape(B, vocab) >> np.uint64(8)
    u = (w.astype(np.float64) + 1.0) * 2.0 ** -24
    key = -np.log(np.maximum(-np.log(u), osm.NOISE_FLOOR))        # logits 0, T 1
    in_order = np.take_along_axis(key, order, axis=1)
    assert np.all(in_order[:, :-1] >= in_order[:, 1:] - 1e-5)
    exact = np.argsort(-w.astype(np.int64), axis=1, kind="stable")
    assert np.mean(np.all(order == exact, axis=1)) >= 0.95
