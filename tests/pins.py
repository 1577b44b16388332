"""Checks that pin the oracle to things other than itself.

Each check takes the implementation under test as an argument, so the same
check runs against the oracle (tests/test_oracle_*.py) and against copies of
the oracle with a planted mistake (tests/test_oracle_mutations.py), which must
make it fail.

The independent references used here:
  * torch.nn.functional.scaled_dot_product_attention in float64 on contiguous
    K/V (a library routine: it knows nothing of paging, block tables or
    prefixes);
  * pure-Python loops with math.exp on tiny inputs;
  * closed forms (one visible key gives V_0; noise 1 gives greedy argmax);
  * the Gumbel-max law P(token k) = softmax(x)_k, tested by chi-square.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import slots as oslots


# ----------------------------------------------------------------------------
# building paged cases from logical, contiguous K/V
# ----------------------------------------------------------------------------
def scatter_logical(K_seqs, V_seqs, block_size, num_blocks, rng):
    """Places each sequence's logical K/V rows into a NaN pool through a random
    block table.  A slot is a flat row index of the pool viewed as
    [num_blocks*block_size, Hkv, D]; the slot list of a sequence is the pages'
    get_slots."""
    Hkv, D = K_seqs[0].shape[1], K_seqs[0].shape[2]
    kpool = np.full((num_blocks * block_size, Hkv, D), np.nan)
    vpool = np.full((num_blocks * block_size, Hkv, D), np.nan)
    perm = list(rng.permutation(num_blocks))
    tables = []
    for K, V in zip(K_seqs, V_seqs):
        n = K.shape[0]
        nb = oslots.num_blocks(n, block_size)
        table = [int(perm.pop()) for _ in range(nb)]
        tables.append(table)
        if n:
            s = oslots.get_slots(table, block_size, n)
            kpool[s] = K
            vpool[s] = V
    width = max(1, max(len(t) for t in tables))
    bt = np.full((len(tables), width), -1, dtype=np.int64)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    shape = (num_blocks, block_size, Hkv, D)
    return kpool.reshape(shape), vpool.reshape(shape), bt


def sdpa_rows(q, K, V, scale, num_cached):
    """Dense reference for one sequence: q (Lq, Hq, D), K/V (Lk, Hkv, D)
    contiguous; query i may see keys j <= num_cached + i.  GQA by repeating each
    kv head over its group of consecutive q heads."""
    Lq, Hq, D = q.shape
    Lk, Hkv, _ = K.shape
    G = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(K).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    vt = torch.from_numpy(V).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    if num_cached == 0 and Lq == Lk:
        o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    else:
        i = torch.arange(Lq)[:, None]
        j = torch.arange(Lk)[None, :]
        o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=(j <= num_cached + i),
                                           scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def random_prefill_case(rng, lens, cached, Hq=4, Hkv=2, D=16, bs=4, spare=3):
    """lens[b] queries after cached[b] cached tokens.  Returns the arguments of
    a prefill call plus the logical per-sequence (q, K, V)."""
    K_all = [rng.standard_normal((c + n, Hkv, D)) for n, c in zip(lens, cached)]
    V_all = [rng.standard_normal((c + n, Hkv, D)) for n, c in zip(lens, cached)]
    Q_all = [rng.standard_normal((n, Hq, D)) for n in lens]
    nb = sum(oslots.num_blocks(c + n, bs) for n, c in zip(lens, cached)) + spare
    # the cache holds only the cached prefixes
    kc, vc, bt = scatter_logical([K[:c] for K, c in zip(K_all, cached)],
                                 [V[:c] for V, c in zip(V_all, cached)], bs, nb, rng)
    # tables must cover the chunk too (its blocks are allocated up front)
    full_nb = [oslots.num_blocks(c + n, bs) for n, c in zip(lens, cached)]
    used = set(int(x) for x in bt.reshape(-1) if x >= 0)
    free = [b for b in range(nb) if b not in used]
    rows = []
    for i in range(len(lens)):
        t = [int(x) for x in bt[i] if x >= 0]
        while len(t) < full_nb[i]:
            t.append(free.pop())
        rows.append(t)
    width = max(len(t) for t in rows)
    bt = np.full((len(rows), width), -1, dtype=np.int64)
    for i, t in enumerate(rows):
        bt[i, :len(t)] = t
    q = np.concatenate(Q_all)
    k = np.concatenate([K[c:] for K, c in zip(K_all, cached)])
    v = np.concatenate([V[c:] for V, c in zip(V_all, cached)])
    cu_q = np.concatenate([[0], np.cumsum(lens)])
    cu_k = np.concatenate([[0], np.cumsum([n + c for n, c in zip(lens, cached)])])
    return dict(q=q, k=k, v=v, k_cache=kc, v_cache=vc, cu_q=cu_q, cu_k=cu_k, bt=bt,
                Q=Q_all, K=K_all, V=V_all)


# ----------------------------------------------------------------------------
# attention pins
# ----------------------------------------------------------------------------
def check_prefill_vs_sdpa(prefill_fn, seed=0, lens=(5, 1, 9, 4), cached=(0, 7, 3, 12),
                          Hq=4, Hkv=2, D=16, bs=4):
    rng = np.random.default_rng(seed)
    c = random_prefill_case(rng, list(lens), list(cached), Hq, Hkv, D, bs)
    scale = 1.0 / math.sqrt(D)
    out = prefill_fn(c["q"], c["k"], c["v"], c["k_cache"], c["v_cache"], c["cu_q"],
                     c["cu_k"], c["bt"], scale)
    for b, (n, cb) in enumerate(zip(lens, cached)):
        ref = sdpa_rows(c["Q"][b], c["K"][b], c["V"][b], scale, cb)
        got = out[c["cu_q"][b]:c["cu_q"][b + 1]]
        assert np.allclose(got, ref, rtol=0, atol=1e-12), f"sequence {b}"


def check_causal_no_cache_vs_sdpa(prefill_fn, seed=1, lens=(6, 11, 1), Hq=2, Hkv=1, D=8):
    """Lq == Lk with no block table: the library's own is_causal path."""
    rng = np.random.default_rng(seed)
    c = random_prefill_case(rng, list(lens), [0] * len(lens), Hq, Hkv, D, bs=4)
    scale = 0.3
    out = prefill_fn(c["q"], c["k"], c["v"], c["k_cache"], c["v_cache"], c["cu_q"],
                     c["cu_k"], None, scale)
    for b in range(len(lens)):
        ref = sdpa_rows(c["Q"][b], c["K"][b], c["V"][b], scale, 0)
        assert np.allclose(out[c["cu_q"][b]:c["cu_q"][b + 1]], ref, rtol=0, atol=1e-12)


def check_decode_vs_sdpa(decode_fn, seed=2, ctx=(1, 5, 17, 32, 0), Hq=8, Hkv=2, D=16, bs=4):
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    V = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    nb = sum(oslots.num_blocks(n, bs) for n in ctx) + 2
    kc, vc, bt = scatter_logical(K, V, bs, nb, rng)
    q = rng.standard_normal((len(ctx), Hq, D))
    scale = 0.25
    out = decode_fn(q, kc, vc, bt, np.array(ctx), scale)
    for b, n in enumerate(ctx):
        if n == 0:
            assert np.all(out[b] == 0.0)
            continue
        ref = sdpa_rows(q[b][None], K[b], V[b], scale, n - 1)[0]
        assert np.allclose(out[b], ref, rtol=0, atol=1e-12), f"sequence {b}"


def check_gather_equals_dense(decode_fn, seed=3, ctx=(13, 29), Hq=4, Hkv=2, D=8, bs=4):
    """The same logical K/V, once scattered through a random block table and
    once laid out contiguously (block i = logical block i): identical outputs."""
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    V = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    q = rng.standard_normal((len(ctx), Hq, D))
    nb = sum(oslots.num_blocks(n, bs) for n in ctx) + 3
    kc, vc, bt = scatter_logical(K, V, bs, nb, rng)
    paged = decode_fn(q, kc, vc, bt, np.array(ctx), 0.5)
    for b, n in enumerate(ctx):
        m = oslots.num_blocks(n, bs)
        kd = np.full((m * bs, Hkv, D), np.nan)
        vd = np.full((m * bs, Hkv, D), np.nan)
        kd[:n], vd[:n] = K[b], V[b]
        dense = decode_fn(q[b:b + 1], kd.reshape(m, bs, Hkv, D), vd.reshape(m, bs, Hkv, D),
                          np.arange(m)[None], np.array([n]), 0.5)
        assert np.array_equal(paged[b], dense[0]), f"sequence {b}"


def check_brute_force_tiny(prefill_fn, seed=4):
    """Pure-Python loops (math.exp, explicit sums) on a tiny GQA case with a
    cached prefix."""
    rng = np.random.default_rng(seed)
    lens, cached, Hq, Hkv, D = [3, 2], [5, 0], 2, 1, 4
    c = random_prefill_case(rng, lens, cached, Hq, Hkv, D, bs=4)
    scale = 0.7
    out = prefill_fn(c["q"], c["k"], c["v"], c["k_cache"], c["v_cache"], c["cu_q"],
                     c["cu_k"], c["bt"], scale)
    for b in range(2):
        Qb, Kb, Vb = c["Q"][b], c["K"][b], c["V"][b]
        for i in range(lens[b]):
            for h in range(Hq):
                kvh = h * Hkv // Hq
                s = []
                for j in range(cached[b] + i + 1):
                    s.append(scale * sum(Qb[i, h, d] * Kb[j, kvh, d] for d in range(D)))
                m = max(s)
                w = [math.exp(x - m) for x in s]
                z = sum(w)
                for d in range(D):
                    ref = sum(w[j] * Vb[j, kvh, d] for j in range(len(w))) / z
                    got = out[c["cu_q"][b] + i, h, d]
                    assert abs(got - ref) <= 1e-12, (b, i, h, d)


def check_single_visible_key(prefill_fn, seed=5):
    """The first query of a sequence with no cached prefix sees only key 0, so
    its output is exactly V_0."""
    rng = np.random.default_rng(seed)
    c = random_prefill_case(rng, [4, 3], [0, 0], 2, 1, 8, bs=4)
    out = prefill_fn(c["q"], c["k"], c["v"], c["k_cache"], c["v_cache"], c["cu_q"],
                     c["cu_k"], c["bt"], 0.9)
    for b in range(2):
        row = c["cu_q"][b]
        for h in range(2):
            assert np.array_equal(out[row, h], c["V"][b][0, 0])


def check_chunked_equals_oneshot(prefill_fn, store_fn, split_points, total, cached_blocks,
                                 bs=4, Hq=4, Hkv=2, D=8, seed=6):
    """One prompt of `total` tokens with `cached_blocks` full blocks already in
    the cache.  Computing it in chunks that end at `split_points` (each chunk's
    K/V stored into the cache before the next) gives the same rows as one call
    over all the uncached tokens."""
    rng = np.random.default_rng(seed)
    c0 = cached_blocks * bs
    K = rng.standard_normal((total, Hkv, D))
    V = rng.standard_normal((total, Hkv, D))
    Q = rng.standard_normal((total, Hq, D))
    nb = oslots.num_blocks(total, bs) + 2
    table = list(rng.permutation(nb)[:oslots.num_blocks(total, bs)])
    slots_all = oslots.get_slots(table, bs, total)
    kc = np.full((nb * bs, Hkv, D), np.nan)
    vc = np.full((nb * bs, Hkv, D), np.nan)
    kc[slots_all[:c0]], vc[slots_all[:c0]] = K[:c0], V[:c0]
    kc, vc = kc.reshape(nb, bs, Hkv, D), vc.reshape(nb, bs, Hkv, D)
    bt = np.array([table])
    one = prefill_fn(Q[c0:], K[c0:], V[c0:], kc, vc, [0, total - c0], [0, total], bt, 0.4)
    got = np.full_like(one, np.nan)
    start = c0
    for end in list(split_points) + [total]:
        n = end - start
        o = prefill_fn(Q[start:end], K[start:end], V[start:end], kc, vc, [0, n], [0, end], bt,
                       0.4)
        got[start - c0:end - c0] = o
        kc, vc = store_fn(K[start:end], V[start:end], kc, vc, slots_all[start:end])
        start = end
    assert np.allclose(got, one, rtol=0, atol=1e-12)


def check_pool_permutation_invariance(decode_fn, seed=7, ctx=(9, 14), Hq=2, Hkv=2, D=8, bs=4):
    """Relabelling the physical blocks (and the tables with them) leaves the
    output unchanged."""
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    V = [rng.standard_normal((n, Hkv, D)) for n in ctx]
    q = rng.standard_normal((len(ctx), Hq, D))
    nb = sum(oslots.num_blocks(n, bs) for n in ctx) + 2
    kc, vc, bt = scatter_logical(K, V, bs, nb, rng)
    a = decode_fn(q, kc, vc, bt, np.array(ctx), 0.3)
    sigma = rng.permutation(nb)                  # new id of old block i is sigma[i]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[sigma], vc2[sigma] = kc, vc
    bt2 = np.where(bt >= 0, sigma[np.maximum(bt, 0)], -1)
    b = decode_fn(q, kc2, vc2, bt2, np.array(ctx), 0.3)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------------------
# sampler pins
# ----------------------------------------------------------------------------
def check_unit_noise_is_greedy(sample_fn, seed=8):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((6, 50)) * 4
    T = np.array([0.2, 0.7, 1.0, 1.5, 3.0, 0.05])
    ids, bad = sample_fn(logits, T, np.ones_like(logits))
    assert not bad
    assert np.array_equal(ids, np.argmax(logits, axis=1))


def check_gumbel_law(sample_fn, seed=9, draws=100_000):
    """Exponential-race / Gumbel-max: the sampled index is distributed as
    softmax(logits / T).  Chi-square goodness of fit over `draws` rows."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(seed)
    row = np.array([1.0, -0.5, 2.0, 0.0, 0.3, -2.0, 1.2, 0.8])
    T = 0.8
    logits = np.tile(row, (draws, 1))
    E = rng.exponential(1.0, size=logits.shape)
    ids, _ = sample_fn(logits, np.full(draws, T), E)
    counts = np.bincount(ids, minlength=row.size)
    p = np.exp(row / T - (row / T).max())
    p /= p.sum()
    _, pval = chisquare(counts, p * draws)
    assert pval > 1e-4, pval


def check_lowest_index_tie(sample_fn):
    logits = np.array([[1.0, 3.0, 3.0, 0.0], [2.0, 2.0, 2.0, 2.0]])
    ids, _ = sample_fn(logits, np.array([1.0, 0.5]), np.ones_like(logits))
    assert ids.tolist() == [1, 0]


def check_temperature_matters(sample_fn):
    """A low temperature lets the largest logit beat noise that a high one
    does not: logits (2, 0), noise (1, 0.3).  Keys x_i - ln E_i:
    T=0.1 -> (20, 1.2) picks 0; T=10 -> (0.2, 1.2) picks 1."""
    logits = np.array([[2.0, 0.0], [2.0, 0.0]])
    E = np.array([[1.0, 0.3], [1.0, 0.3]])
    ids, _ = sample_fn(logits, np.array([0.1, 10.0]), E)
    assert ids.tolist() == [0, 1]


# ----------------------------------------------------------------------------
# counter-based generator pin
# ----------------------------------------------------------------------------
def philox_kat_cases():
    """The known-answer cases of tests/golden/philox4x32_10_kat.json as
    (counter words, key words, output words) integer tuples."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "philox4x32_10_kat.json")
    gold = json.load(open(path))
    assert gold["rounds"] == 10
    return [(tuple(int(x, 16) for x in c["counter"]), tuple(int(x, 16) for x in c["key"]),
             tuple(int(x, 16) for x in c["output"])) for c in gold["cases"]]


def check_philox_kat(block_fn):
    """block_fn(counters (N, 4), key (k0, k1)) -> (N, 4) words must reproduce
    the published Philox4x32-10 known-answer vectors word for word."""
    for ctr, key, want in philox_kat_cases():
        got = block_fn(np.array([ctr], dtype=np.uint64), key)
        assert [int(x) for x in np.asarray(got)[0]] == list(want), (ctr, key)
