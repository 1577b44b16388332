"""Attention over a paged KV cache, restated on the CPU in float64.

Test infrastructure only (see the package docstring).

Layouts ([UML] §3.2 "Attention运算"; [LIFE] §2.2.3):
  q                 (num_tokens, Hq, D)
  k, v              (num_tokens, Hkv, D)
  k_cache, v_cache  (num_blocks, block_size, Hkv, D) -- one layer's view of the pool
  block_tables      (batch, max_blocks_per_seq), logical block -> physical block
  cu_seqlens_q/k    (batch+1,) prefix sums of per-sequence lengths
  context_lens      (batch,) cached keys per sequence (decode)

Readings where the pages are silent:
  * grouped-query attention maps q head h to kv head h // (Hq // Hkv);
  * a query that is row i of a sequence with Lq queries and Lk keys sits at
    absolute position Lk - Lq + i and sees keys j <= that position (the only
    alignment under which a chunked prefill equals a one-shot one);
  * in prefill the first Lk - Lq keys (the cached prefix) are read through the
    block table and the last Lq keys are the call's own k / v rows;
  * the decode context length counts the token being decoded (its K/V are
    stored before attention runs, [LIFE] §2.2.4 layer op order);
  * a sequence with no keys produces zeros.

Inputs may be NumPy arrays or CPU torch tensors (bf16 caches are widened to
float64 only for the rows a sequence uses); every product and sum below is
float64.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):                       # a torch tensor
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _take(cache, blocks: np.ndarray, rows: np.ndarray, head: int) -> np.ndarray:
    if hasattr(cache, "detach"):
        import torch
        sub = cache[torch.as_tensor(blocks, dtype=torch.long),
                    torch.as_tensor(rows, dtype=torch.long), head]
        return _f64(sub)
    return _f64(np.asarray(cache)[blocks, rows, head])


def gather_keys(cache, block_table, num_keys: int, kv_head: int) -> np.ndarray:
    """The logical key (or value) list of one sequence and kv head: entry j is
    row j % block_size of physical block block_table[j // block_size]
    ([UML] §1 Step2 slot formula; §2.1 block table: logical block i maps to a
    physical block that need not be contiguous)."""
    num_blocks, block_size = cache.shape[0], cache.shape[1]
    if num_keys == 0:
        return np.zeros((0, cache.shape[3]))
    j = np.arange(num_keys)
    table = np.asarray(block_table).reshape(-1)
    blocks = table[j // block_size]
    if blocks.min() < 0 or blocks.max() >= num_blocks:
        raise ValueError("block table entry outside the pool")
    return _take(cache, blocks, j % block_size, kv_head)


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Grouped-query attention (named, not defined, in [LIFE] §3.3.2): the kv
    cache stores Hkv heads only ([LIFE] §2.2.3 block_bytes counts num_kv_heads)
    and q head h reads kv head h // (Hq // Hkv) -- contiguous groups."""
    return h // (num_q_heads // num_kv_heads)


def query_positions(num_q: int, num_k: int) -> np.ndarray:
    """Absolute positions of a sequence's queries: the Lq queries are the last
    Lq of its Lk tokens, so query i sits at Lk - Lq + i ([LIFE] §3.1: a round
    computes num_scheduled_tokens tokens starting at num_cached_tokens)."""
    return (num_k - num_q) + np.arange(num_q)


def attend(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray,
           scale: float, positions) -> np.ndarray:
    """Softmax attention, the plain definition: query row r with absolute
    position p_r gets sum_j softmax_j(scale * q_r . K_j) V_j over keys j <= p_r,
    with the usual subtraction of the row maximum before exp."""
    L = keys.shape[0]
    s = scale * (q_rows @ keys.T)
    visible = np.arange(L)[None, :] <= np.asarray(positions)[:, None]
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.where(visible, np.exp(s - m), 0.0)
    return (e @ values) / e.sum(axis=1, keepdims=True)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 seqs=None, heads=None) -> np.ndarray:
    """Decode attention ([UML] §2.4: the decode FA op reads K/V through
    block_tables with cache_seqlens; §3.2 formats): one query per sequence,
    attending all context_lens[b] cached keys.  Returns (B, Hq, D) float64;
    rows of sequences not listed in `seqs` are NaN, and so are the q heads of
    sequence b not listed in heads(b) when `heads` (a function of b) is given."""
    qf = _f64(q)
    B, Hq, D = qf.shape
    Hkv = k_cache.shape[2]
    bt = np.asarray(block_tables)
    ctx = np.asarray(context_lens).reshape(-1)
    out = np.full((B, Hq, D), np.nan)
    for b in (range(B) if seqs is None else seqs):
        n = int(ctx[b])
        hs = range(Hq) if heads is None else heads(b)
        if n == 0:
            out[b, list(hs)] = 0.0
            continue
        for h in hs:
            kvh = kv_head_of(h, Hq, Hkv)
            K = gather_keys(k_cache, bt[b], n, kvh)
            V = gather_keys(v_cache, bt[b], n, kvh)
            out[b, h] = attend(qf[b, h][None], K, V, scale, query_positions(1, n))[0]
    return out


def paged_prefill_varlen(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k,
                         block_tables, scale: float, rows=None) -> np.ndarray:
    """Causal varlen prefill over a prefix-cached paged cache ([UML] §2.4 and
    §3.2: the prefill FA op with cu_seqlens_q/k and, when a prefix is cached,
    block_tables; [LIFE] §3.1 / [SRC2]: a chunk computes num_scheduled_tokens
    tokens starting at num_cached_tokens).

    Sequence b has Lq = cu_q[b+1]-cu_q[b] queries and Lk = cu_k[b+1]-cu_k[b]
    keys.  Keys j < Lk-Lq come from the cache through block_tables[b]; keys
    j >= Lk-Lq are rows cu_q[b] + (j - (Lk-Lq)) of k / v.  Query i sits at
    position Lk-Lq+i.

    `rows` optionally maps b -> iterable of query indices i to compute; the
    other output rows are NaN.  Returns (total_q, Hq, D) float64."""
    qf = _f64(q)
    T, Hq, D = qf.shape
    Hkv = k.shape[1]
    cu_q = np.asarray(cu_seqlens_q).reshape(-1)
    cu_k = np.asarray(cu_seqlens_k).reshape(-1)
    out = np.full((T, Hq, D), np.nan)
    B = len(cu_q) - 1
    for b in range(B):
        if rows is not None and b not in rows:
            continue
        q0, Lq = int(cu_q[b]), int(cu_q[b + 1] - cu_q[b])
        Lk = int(cu_k[b + 1] - cu_k[b])
        c = Lk - Lq
        if Lq == 0:
            continue
        if c < 0:
            raise ValueError("a sequence has fewer keys than queries")
        if c > 0 and block_tables is None:
            raise ValueError("a cached prefix needs block_tables")
        sel = np.arange(Lq) if rows is None else np.asarray(sorted(rows[b]), dtype=np.int64)
        pos = query_positions(Lq, Lk)[sel]
        for h in range(Hq):
            kvh = kv_head_of(h, Hq, Hkv)
            parts_k, parts_v = [], []
            if c > 0:
                bt = np.asarray(block_tables)[b]
                parts_k.append(gather_keys(k_cache, bt, c, kvh))
                parts_v.append(gather_keys(v_cache, bt, c, kvh))
            parts_k.append(_f64(k[q0:q0 + Lq, kvh]))
            parts_v.append(_f64(v[q0:q0 + Lq, kvh]))
            K, V = np.concatenate(parts_k), np.concatenate(parts_v)
            out[q0 + sel, h] = attend(qf[q0 + sel, h], K, V, scale, pos)
    return out
