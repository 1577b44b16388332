"""Slot arithmetic of the oracle against the values the pages print."""
import json
import os

import numpy as np

from oracle import kv_store as okv
from oracle import slots as oslots

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "slot_examples.json")))


def test_slot_formula_worked_example():
    g = GOLD["slot_formula"]
    assert oslots.slot_of(g["block_id"], g["block_size"], g["loc"]) == g["slot"]


def test_prepare_prefill_example():
    g = GOLD["prepare_prefill_example"]
    seqs = [(s["num_cached_tokens"], s["num_scheduled_tokens"], s["block_table"]) for s in g["seqs"]]
    positions, cu_q, cu_k, slots = oslots.prefill_metadata(seqs, g["block_size"])
    assert positions == g["positions"]
    assert cu_q == g["cu_seqlens_q"]
    assert cu_k == g["cu_seqlens_q"]          # nothing cached: k lengths equal q lengths
    assert slots == g["slot_mapping"]


def test_get_slots_matches_prepare_prefill_example():
    g = GOLD["prepare_prefill_example"]
    flat = []
    for s in g["seqs"]:
        flat += oslots.get_slots(s["block_table"], g["block_size"], s["num_scheduled_tokens"])
    assert flat == g["slot_mapping"]


def test_sequence_counter_walkthrough():
    g = GOLD["sequence_counter_walkthrough"]
    bs, n = g["block_size"], g["num_tokens"]
    assert oslots.num_blocks(n, bs) == g["num_blocks"]
    assert oslots.last_block_num_tokens(n, bs) == g["last_block_num_tokens"]
    rounds = oslots.chunk_rounds(n, g["cached_blocks"] * bs, g["budget"])
    assert [list(r) for r in rounds] == g["rounds"]
    after = np.cumsum([c for _, c in rounds]) + g["cached_blocks"] * bs
    assert after.tolist() == g["num_cached_tokens_after_round"]
    slots = oslots.get_slots(g["block_table"], bs, n)
    per_block = [sum(1 for s in slots if s // bs == b) for b in g["block_table"]]
    assert per_block == g["tokens_per_block"]
    assert slots[0] == 5 * 256 and slots[256] == 9 * 256 and slots[-1] == 12 * 256 + 87


def test_get_slots_equals_slot_of_each_position():
    rng = np.random.default_rng(0)
    for bs in (1, 4, 16, 256):
        for n in (1, bs - 1 if bs > 1 else 1, bs, bs + 1, 3 * bs + 5):
            table = list(rng.permutation(100)[:oslots.num_blocks(n, bs)])
            s = oslots.get_slots(table, bs, n)
            assert len(s) == n and len(set(s)) == n
            assert s == [oslots.slot_of(table[p // bs], bs, p % bs) for p in range(n)]


def test_block_growth_only_when_full():
    # 7 tokens in 2 blocks of 4; appending tokens 8..14: a block is added when
    # the token count reaches 9 and 13 (the last block was full)
    grows = [n for n in range(8, 15) if oslots.needs_new_block(n, oslots.num_blocks(n - 1, 4), 4)]
    assert grows == [9, 13]
    assert oslots.decode_slot([7, 3, 2], 9, 4) == 2 * 4 + 0


def test_kv_store_bruteforce_and_102():
    rng = np.random.default_rng(1)
    nb, bs, hkv, d = 30, 4, 2, 3
    kc = rng.integers(0, 2**16, size=(nb, bs, hkv, d), dtype=np.uint16)
    vc = rng.integers(0, 2**16, size=(nb, bs, hkv, d), dtype=np.uint16)
    k = rng.integers(0, 2**16, size=(5, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 2**16, size=(5, hkv, d), dtype=np.uint16)
    slots = np.array([102, -1, 0, 119, 7])
    k2, v2, bad = okv.kv_store(k, v, kc, vc, slots)
    assert bad == []
    assert np.array_equal(k2[25, 2], k[0]) and np.array_equal(v2[25, 2], v[0])  # 25*4+2
    flat_k, flat_v = kc.reshape(nb * bs, hkv, d).copy(), vc.reshape(nb * bs, hkv, d).copy()
    for i, s in enumerate(slots):
        if s >= 0:
            flat_k[s], flat_v[s] = k[i], v[i]
    assert np.array_equal(k2.reshape(nb * bs, hkv, d), flat_k)
    assert np.array_equal(v2.reshape(nb * bs, hkv, d), flat_v)
    # out-of-range slots are reported and skipped
    k3, _, bad = okv.kv_store(k[:1], v[:1], kc, vc, np.array([nb * bs]))
    assert bad == [nb * bs] and np.array_equal(k3, kc)
