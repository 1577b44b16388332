"""sample on the GPU against the oracle: identical token ids (near-ties, where
float32 and float64 may legitimately differ, accept any near-top index and are
counted)."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import sampler as osm
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check(pkv, logits, temps, noise, dev, expect_status=0):
    st = pkv.new_status(dev)
    ids = pkv.sample(logits.to(dev), temps.to(dev), noise.to(dev), status=st).cpu().numpy()
    ref, bad = osm.sample(logits.numpy(), temps.numpy(), noise.numpy())
    ref2, keys = osm.sample_key_form(logits.numpy(), temps.numpy(), noise.numpy())
    assert np.array_equal(ref, ref2)
    near = osm.near_ties(keys)
    ambiguous = 0
    for r in range(len(ids)):
        if r in bad:
            assert ids[r] == 0
        elif len(near[r]) > 1:
            ambiguous += 1
            assert ids[r] in near[r], (r, ids[r], near[r])
        else:
            assert ids[r] == ref[r], (r, ids[r], ref[r])
    assert U.status_word(st) == expect_status
    return ambiguous


def test_tiny_vocab_1000(cuda):
    pkv = U.lib()
    w = W.tiny_workload()
    assert _check(pkv, w.logits, w.temperatures, w.exp_noise, cuda) == 0


def test_step_8b_full_vocab(cuda):
    pkv = U.lib()
    g = torch.Generator().manual_seed(4)
    logits, temps, noise = W.sampler_inputs(512, 151936, 3.0, 4, 0.2, 1.2, g)
    amb = _check(pkv, logits, temps, noise, cuda)
    print(f"ambiguous rows: {amb} of 512")


@pytest.mark.parametrize("vocab", [1, 7, 1001, 16385, 131073])
def test_ragged_vocab_sizes(cuda, vocab):
    pkv = U.lib()
    g = torch.Generator().manual_seed(vocab)
    logits, temps, noise = W.sampler_inputs(9, vocab, 2.0, 0, 0.5, 1.5, g)
    _check(pkv, logits, temps, noise, cuda)


def test_unit_noise_is_greedy_and_ties_take_lowest_index(cuda):
    pkv = U.lib()
    logits = torch.zeros((3, 4099), dtype=torch.float32)
    logits[0, 17] = 5.0
    logits[1, 4000] = 2.0
    logits[1, 4001] = 2.0
    logits[1, 100] = 2.0                     # ties: lowest index wins
    temps = torch.tensor([0.3, 1.0, 2.0])
    ids = pkv.sample(logits.to(cuda), temps.to(cuda), torch.ones_like(logits).to(cuda)).cpu()
    assert ids.tolist() == [17, 100, 0]


def test_bad_temperature_rows(cuda):
    pkv = U.lib()
    g = torch.Generator().manual_seed(5)
    logits, _, noise = W.sampler_inputs(4, 300, 1.0, 0, 1.0, 1.0, g)
    temps = torch.tensor([1.0, 0.0, -2.0, float("nan")])
    _check(pkv, logits, temps, noise, cuda, expect_status=pkv.STATUS["BAD_TEMPERATURE"])
