"""The attention oracle against a library routine, brute force and closed forms."""
import numpy as np

import pins
from oracle import attention as oatt
from oracle import kv_store as okv


def _store(k, v, kc, vc, s):
    a, b, _ = okv.kv_store(k, v, kc, vc, np.asarray(s))
    return a, b


def test_prefill_vs_sdpa_with_cached_prefix():
    pins.check_prefill_vs_sdpa(oatt.paged_prefill_varlen)


def test_prefill_vs_sdpa_mha_and_group4():
    pins.check_prefill_vs_sdpa(oatt.paged_prefill_varlen, seed=11, Hq=3, Hkv=3)
    pins.check_prefill_vs_sdpa(oatt.paged_prefill_varlen, seed=12, Hq=8, Hkv=2, bs=16,
                               lens=(20, 3), cached=(33, 16))


def test_causal_without_block_table_vs_sdpa():
    pins.check_causal_no_cache_vs_sdpa(oatt.paged_prefill_varlen)


def test_decode_vs_sdpa():
    pins.check_decode_vs_sdpa(oatt.paged_decode)


def test_gather_through_random_table_equals_dense():
    pins.check_gather_equals_dense(oatt.paged_decode)


def test_bruteforce_tiny():
    pins.check_brute_force_tiny(oatt.paged_prefill_varlen)


def test_single_visible_key_is_v0():
    pins.check_single_visible_key(oatt.paged_prefill_varlen)


def test_chunked_equals_oneshot_at_walkthrough_points():
    # 600-token prompt, one cached 256-token block, budget 200: chunks end at 456
    pins.check_chunked_equals_oneshot(oatt.paged_prefill_varlen, _store, [456], 600, 1, bs=256)


def test_chunked_equals_oneshot_random_points():
    rng = np.random.default_rng(3)
    for trial in range(3):
        total = int(rng.integers(20, 60))
        cached = int(rng.integers(0, 3))
        pts = sorted(set(int(x) for x in rng.integers(cached * 4 + 1, total, size=3)))
        pins.check_chunked_equals_oneshot(oatt.paged_prefill_varlen, _store, pts, total,
                                          cached, bs=4, seed=trial)


def test_pool_permutation_invariance():
    pins.check_pool_permutation_invariance(oatt.paged_decode)


def test_decode_equals_prefill_with_one_query():
    rng = np.random.default_rng(4)
    c = pins.random_prefill_case(rng, [1, 1, 1], [9, 0, 30], Hq=4, Hkv=2, D=8, bs=4)
    pre = oatt.paged_prefill_varlen(c["q"], c["k"], c["v"], c["k_cache"], c["v_cache"],
                                    c["cu_q"], c["cu_k"], c["bt"], 0.5)
    # store the single new token of each sequence, then decode over all keys
    slots = [pins.oslots.decode_slot(list(c["bt"][b][c["bt"][b] >= 0]), n + 1, 4)
             for b, n in enumerate([9, 0, 30])]
    kc, vc = _store(c["k"], c["v"], c["k_cache"], c["v_cache"], slots)
    dec = oatt.paged_decode(c["q"], kc, vc, c["bt"], np.array([10, 1, 31]), 0.5)
    assert np.allclose(pre, dec, rtol=0, atol=1e-12)
