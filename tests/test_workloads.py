"""The seeded generators: determinism, poison, and engine-side metadata checked
against the oracle's independent slot arithmetic."""
import numpy as np
import torch

from oracle import slots as oslots
from paged_kv_attention_scatter_gb300 import workloads as W


def test_tiny_scenario_matches_slot_rules():
    w = W.tiny_workload()
    p = w.prefill
    tables = [list(t[t >= 0].tolist()) for t in p.block_tables]
    _, cu_q, cu_k, slots = oslots.prefill_metadata([(0, 7, tables[0]), (0, 11, tables[1])], 4)
    assert p.cu_seqlens_q.tolist() == cu_q and p.cu_seqlens_k.tolist() == cu_k
    assert p.slot_mapping.tolist() == slots
    # three decode steps: contexts 8,9,10 and 12,13,14; blocks appended at 9 and 13
    assert [s.context_lens.tolist() for s in w.decode_steps] == [[8, 12], [9, 13], [10, 14]]
    for s in w.decode_steps:
        for i in range(2):
            t = s.block_tables[i][s.block_tables[i] >= 0].tolist()
            n = int(s.context_lens[i])
            assert len(t) == oslots.num_blocks(n, 4)
            assert int(s.slot_mapping[i]) == oslots.decode_slot(t, n, 4)
    used = set(b for t in w.block_tables_final for b in t)
    assert len(used) == 7 and used <= set(range(8))
    assert w.temperatures.tolist() == [0.699999988079071, 1.0]


def test_decode_workload_layout_and_poison():
    spec = W.DecodeSpec("t", seed=5, batch=6, num_q_heads=4, num_kv_heads=2, head_dim=8,
                        block_size=4, ctx_lo=1, ctx_hi=13, store_new_token=True,
                        vocab=50, logit_spikes=2, t_lo=0.2, t_hi=1.2)
    a = W.decode_workload(spec)
    b = W.decode_workload(spec)
    assert torch.equal(a.q, b.q) and torch.equal(a.block_tables, b.block_tables)
    kc = a.k_cache.float()
    nb, bs = kc.shape[:2]
    valid = np.zeros((nb, bs), bool)
    for i in range(spec.batch):
        n = int(a.context_lens[i])
        t = a.block_tables[i][a.block_tables[i] >= 0].tolist()
        assert len(t) == oslots.num_blocks(n, bs)
        s = oslots.get_slots(t, bs, n)
        assert int(a.slot_mapping[i]) == s[-1] == oslots.decode_slot(t, n, bs)
        for x in s[:-1]:                        # held before the step
            valid[x // bs, x % bs] = True
    assert torch.isfinite(kc[torch.from_numpy(valid)]).all()
    assert torch.isnan(kc[torch.from_numpy(~valid)]).all()
    assert a.logits.shape == (6, 50) and (a.exp_noise > 0).all()
    assert ((a.temperatures >= 0.2) & (a.temperatures <= 1.2)).all()


def test_prefill_workload_chunks():
    spec = W.PrefillSpec("t", seed=7, num_prompts=5, num_q_heads=4, num_kv_heads=2,
                         head_dim=8, block_size=16, len_lo=20, len_hi=90,
                         max_cached_blocks=3, token_budget=64)
    w = W.prefill_workload(spec)
    bs = spec.block_size
    done = [kb * bs for kb in w.cached_blocks]
    for st in w.steps[:-1]:
        assert st.q.shape[0] == spec.token_budget
    for st in w.steps:
        cu_q, cu_k = st.cu_seqlens_q.tolist(), st.cu_seqlens_k.tolist()
        seqs = []
        for j, r in enumerate(st.seq_ids):
            lq, lk = cu_q[j + 1] - cu_q[j], cu_k[j + 1] - cu_k[j]
            assert lk - lq == done[r] == st.q_start[j]
            seqs.append((done[r], lq, w.block_tables[r]))
            done[r] += lq
        _, cq, ck, sl = oslots.prefill_metadata(seqs, bs)
        assert cq == cu_q and ck == cu_k and st.slot_mapping.tolist() == sl
    assert done == w.prompt_lens
    # prompts share their cached prefix blocks
    pre = [t[:kb] for t, kb in zip(w.block_tables, w.cached_blocks)]
    longest = max(pre, key=len)
    assert all(p == longest[:len(p)] for p in pre)


def test_mixed_workload_metadata_and_poison():
    """A continuous-batching step: decode rows (one new token at ctx-1) first,
    then prefill chunks; its varlen metadata follows the same slot rules, each
    decode row's new token lands at its context's last position, and only the
    cached tokens of the pool hold numbers."""
    import dataclasses
    spec = dataclasses.replace(W.MIXED_8B, num_decode=6, num_prefill=3, num_q_heads=4,
                               num_kv_heads=2, head_dim=8, block_size=16, ctx_lo=1,
                               ctx_hi=70, new_lo=2, new_hi=40, cached_lo=0, cached_hi=50)
    w = W.mixed_workload(spec)
    st, bs = w.step, spec.block_size
    cu_q, cu_k = st.cu_seqlens_q.tolist(), st.cu_seqlens_k.tolist()
    tables = [[int(x) for x in row if x >= 0] for row in st.block_tables]
    seqs = []
    for j in range(len(cu_q) - 1):
        lq, lk = cu_q[j + 1] - cu_q[j], cu_k[j + 1] - cu_k[j]
        assert (lq == 1) == (j < spec.num_decode)
        assert lk - lq == st.q_start[j]
        assert len(tables[j]) == oslots.num_blocks(lk, bs)
        if lq == 1:
            assert st.slot_mapping[cu_q[j]] == oslots.decode_slot(tables[j], lk, bs)
        seqs.append((lk - lq, lq, tables[j]))
    _, cq, ck, sl = oslots.prefill_metadata(seqs, bs)
    assert cq == cu_q and ck == cu_k and st.slot_mapping.tolist() == sl
    # every block belongs to one sequence; cached rows hold numbers, the rest NaN
    flat = sorted(b for t in tables for b in t)
    assert flat == list(range(w.k_cache0.shape[0]))
    for t, (cached, _, _) in zip(tables, seqs):
        for pos in range(len(t) * bs):
            row = w.k_cache0[t[pos // bs], pos % bs]
            assert bool(torch.isnan(row).all()) == (pos >= cached)


def test_chunk_plan_walkthrough_and_flag():
    # one 600-token prompt with 256 cached: new tokens 344 at budget 200
    assert W.chunk_plan([344], 200, False) == [[(0, 0, 200)], [(0, 200, 144)]]
    # the pages' rule: only the first sequence of a step may be chunked
    assert W.chunk_plan([100, 150], 200, True) == [[(0, 0, 100)], [(1, 0, 150)]]
    assert W.chunk_plan([100, 150], 200, False) == [[(0, 0, 100), (1, 0, 100)], [(1, 100, 50)]]
