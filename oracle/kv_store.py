"""The KV-cache scatter ("store_kvcache"), restated on the CPU.

Test infrastructure only (see the package docstring).
"""
from __future__ import annotations

import numpy as np


def kv_store(k, v, k_cache, v_cache, slot_mapping):
    """[LIFE] §3.3.2 and §4: slot_mapping[i] is the physical slot of the i-th
    flattened token, and the cache writer needs no other paging knowledge;
    [UML] §2.4 / §3.2: each token's K and V rows go into k_cache / v_cache at
    that slot.  A slot s names block s // block_size, row s % block_size
    ([UML] §1 Step2 formula read backwards).

    k, v: (N, Hkv, D) arrays of any dtype (bf16 data is passed as its raw
    16-bit patterns, so the copy is bit-exact).  k_cache, v_cache:
    (num_blocks, block_size, Hkv, D) of the same dtype.  A negative slot means
    "no token" (a padding row) and is skipped.  Returns new caches and the list
    of slots that were out of range (also skipped)."""
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    num_blocks, block_size = k_out.shape[0], k_out.shape[1]
    bad = []
    for i, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        if s >= num_blocks * block_size:
            bad.append(s)
            continue
        blk, off = s // block_size, s % block_size
        k_out[blk, off] = k[i]
        v_out[blk, off] = v[i]
    return k_out, v_out, bad
