"""GB300-native attention over a paged KV cache.

Four operations, each a hand-written sm_103a CUDA kernel behind the C ABI in
include/pagedattn.h (libpagedattn.so), reached from Python through a thin
ctypes binding:

  kv_store              scatter new K/V rows into cache slots (slot_mapping)
  paged_decode          split-KV decode attention through block tables
  paged_prefill_varlen  causal varlen prefill over a prefix-cached paged cache
  sample                temperature / softmax / Gumbel-max token sampling

PyTorch supplies device memory and streams only.  `workloads` draws the seeded
synthetic inputs the tests and the benchmark use.
"""
from ._binding import (STATUS, cache_desc, kv_store, kv_store_paged_attention_varlen,  # noqa: F401,E501
                       kv_store_paged_decode, kv_store_paged_prefill_varlen,
                       paged_attention_varlen_workspace_bytes, layer_cache, library_path, load,
                       new_status, paged_decode, paged_decode_plan, paged_decode_run,
                       paged_decode_workspace_bytes, paged_prefill_varlen,
                       paged_prefill_workspace_bytes, sample, sample_philox,
                       set_wait_poll_limit, status_names)
from ._build import build  # noqa: F401

__all__ = ["kv_store", "paged_decode", "paged_prefill_varlen", "sample", "build", "load",
           "kv_store_paged_decode", "kv_store_paged_prefill_varlen", "layer_cache",
           "kv_store_paged_attention_varlen", "paged_attention_varlen_workspace_bytes",
           "paged_decode_plan", "paged_decode_run", "sample_philox",
           "paged_decode_workspace_bytes", "paged_prefill_workspace_bytes", "new_status",
           "status_names", "STATUS", "cache_desc", "library_path", "set_wait_poll_limit"]
