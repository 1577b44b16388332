"""Planted mistakes: each test swaps one piece of the oracle for a plausible
wrong version (on the CPU, in this process only) and requires that at least one
pin catches it.  This shows the pins constrain the oracle rather than restate
it."""
import numpy as np
import pytest

import pins
from oracle import attention as oatt
from oracle import kv_store as okv
from oracle import sampler as osm


def _fails(check, *args, **kw):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check(*args, **kw)


def _store(k, v, kc, vc, s):
    a, b, _ = okv.kv_store(k, v, kc, vc, np.asarray(s))
    return a, b


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "kv_head_of", lambda h, hq, hkv: h % hkv)
    _fails(pins.check_prefill_vs_sdpa, oatt.paged_prefill_varlen)
    _fails(pins.check_decode_vs_sdpa, oatt.paged_decode)


def test_top_left_causal_alignment_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "query_positions", lambda nq, nk: np.arange(nq))
    _fails(pins.check_prefill_vs_sdpa, oatt.paged_prefill_varlen)
    _fails(pins.check_chunked_equals_oneshot, oatt.paged_prefill_varlen, _store, [456], 600, 1,
           bs=256)


def test_transposed_block_lookup_is_caught(monkeypatch):
    def bad_gather(cache, table, n, kvh):
        bs = cache.shape[1]
        j = np.arange(n)
        t = np.asarray(table).reshape(-1)
        return oatt._take(cache, t[np.minimum(j % bs, len(t) - 1)], np.minimum(j // bs, bs - 1),
                          kvh)
    monkeypatch.setattr(oatt, "gather_keys", bad_gather)
    _fails(pins.check_decode_vs_sdpa, oatt.paged_decode)
    _fails(pins.check_gather_equals_dense, oatt.paged_decode)


def test_dropped_scale_is_caught(monkeypatch):
    real = oatt.attend
    monkeypatch.setattr(oatt, "attend", lambda q, K, V, s, p: real(q, K, V, 1.0, p))
    _fails(pins.check_brute_force_tiny, oatt.paged_prefill_varlen)


def test_off_by_one_context_is_caught(monkeypatch):
    real = oatt.gather_keys
    monkeypatch.setattr(oatt, "gather_keys",
                        lambda c, t, n, h: real(c, t, max(n - 1, 1), h))
    _fails(pins.check_decode_vs_sdpa, oatt.paged_decode)


def test_swapped_slot_split_is_caught():
    def bad_store(k, v, kc, vc, slots):
        ko, vo = np.array(kc, copy=True), np.array(vc, copy=True)
        bs = ko.shape[1]
        for i, s in enumerate(np.asarray(slots).tolist()):
            if s >= 0:
                ko[s % ko.shape[0], (s // ko.shape[0]) % bs] = k[i]
                vo[s % vo.shape[0], (s // vo.shape[0]) % bs] = v[i]
        return ko, vo
    _fails(pins.check_chunked_equals_oneshot, oatt.paged_prefill_varlen, bad_store, [10, 17], 30,
           2, bs=4)


def _mutant_sampler(kind):
    def sample(logits, temperatures, exp_noise):
        lg = np.asarray(logits, dtype=np.float64)
        T = np.asarray(temperatures, dtype=np.float64)
        E = np.asarray(exp_noise, dtype=np.float64)
        out = np.zeros(lg.shape[0], dtype=np.int32)
        for r in range(lg.shape[0]):
            x = lg[r] / (1.0 if kind == "no_temperature" else T[r])
            p = np.exp(x - x.max())
            p /= p.sum()
            key = p * E[r] if kind == "times_noise" else p / E[r]
            out[r] = int(np.argmax(key)) if kind != "last_tie" else \
                len(key) - 1 - int(np.argmax(key[::-1]))
        return out, []
    return sample


def test_sampler_mutants_are_caught():
    _fails(pins.check_gumbel_law, _mutant_sampler("times_noise"))
    _fails(pins.check_temperature_matters, _mutant_sampler("no_temperature"))
    _fails(pins.check_lowest_index_tie, _mutant_sampler("last_tie"))
    pins.check_gumbel_law(osm.sample)


def _mutant_philox(kind):
    """Philox4x32 block functions with one plausible slip each."""
    M0, M1 = osm.PHILOX_M
    W0, W1 = osm.PHILOX_W
    if kind == "swapped_multipliers":
        M0, M1 = M1, M0
    if kind == "swapped_weyl":
        W0, W1 = W1, W0
    rounds = 7 if kind == "seven_rounds" else 10

    def block(counters, key):
        out = []
        for c0, c1, c2, c3 in np.asarray(counters, dtype=np.uint64).tolist():
            k0, k1 = int(key[0]), int(key[1])
            for r in range(rounds):
                if r > 0 or kind == "bump_before_first":
                    k0, k1 = (k0 + W0) & osm.MASK32, (k1 + W1) & osm.MASK32
                p0, p1 = M0 * c0, M1 * c2
                hi0, lo0 = p0 >> 32, p0 & osm.MASK32
                hi1, lo1 = p1 >> 32, p1 & osm.MASK32
                if kind == "hi_lo_swapped":
                    hi0, lo0, hi1, lo1 = lo0, hi0, lo1, hi1
                if kind == "key_words_swapped":
                    c0, c1, c2, c3 = hi1 ^ c1 ^ k1, lo1, hi0 ^ c3 ^ k0, lo0
                else:
                    c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
            out.append([c0, c1, c2, c3])
        return np.array(out, dtype=np.uint64)
    return block


@pytest.mark.parametrize("kind", ["swapped_multipliers", "swapped_weyl", "seven_rounds",
                                  "bump_before_first", "hi_lo_swapped", "key_words_swapped"])
def test_philox_mutants_are_caught(kind):
    _fails(pins.check_philox_kat, _mutant_philox(kind))


def test_philox_mutant_harness_is_faithful():
    # the mutant factory with no slip is the generator itself
    pins.check_philox_kat(_mutant_philox("none"))
