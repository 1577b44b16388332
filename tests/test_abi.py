"""The C ABI library builds for sm_103a, loads, and exports every symbol the
header declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_scatter_gb300 import _binding, _build
    _build.build()
    return _binding.load()


def test_header_declares_the_four_operations():
    names = declared_functions()
    for op in ("pkv_kv_store", "pkv_paged_decode", "pkv_paged_prefill_varlen", "pkv_sample"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    from paged_kv_attention_scatter_gb300 import _binding
    assert sorted(_binding.C_FUNCTIONS) == declared_functions()


def test_version_and_strings(lib):
    assert lib.pkv_version() >= 100
    assert lib.pkv_error_string(0) == b"ok"
    assert b"null" in lib.pkv_error_string(-1)
    assert lib.pkv_status_string(0) == b"ok"
    assert b"slot" in lib.pkv_status_string(1)


def test_workspace_queries_are_pure(lib):
    from paged_kv_attention_scatter_gb300._binding import CacheDesc
    c = CacheDesc(610, 256, 8, 128)
    a = lib.pkv_paged_decode_workspace_bytes(64, 16, 4096, c)
    assert a == lib.pkv_paged_decode_workspace_bytes(64, 16, 4096, c) and a > 0
    assert lib.pkv_paged_decode_workspace_bytes(64, 16, 8192, c) >= a
    p = lib.pkv_paged_prefill_workspace_bytes(16, 16384, 32, c)
    assert p >= 8 * (16384 // 128 + 16)       # one (sequence, 128-query tile) pair each
    # the mixed-batch call holds the prefill's schedule and a decode plan
    m = lib.pkv_paged_attention_varlen_workspace_bytes(16, 16384, 32, 8192, c)
    assert m >= p + lib.pkv_paged_decode_workspace_bytes(16, 32, 8192, c)
    assert m == lib.pkv_paged_attention_varlen_workspace_bytes(16, 16384, 32, 8192, c)
    assert lib.pkv_paged_attention_varlen_workspace_bytes(16, 16384, 0, 8192, c) == 0


def test_decode_workspace_follows_the_chunk_choice(lib):
    """decode-0.6b (64 sequences, 16/8 heads, D=128, max context 4096): 448-key
    chunks (the multiple of 64 nearest ~16 units per SM), so 10 chunk slots per
    sequence; the workspace is the chunk prefix, the records, the (max, sum)
    pairs and the fp32 partial outputs, each 256-byte aligned."""
    from paged_kv_attention_scatter_gb300._binding import CacheDesc
    cap = 64 * -(-4096 // 448)
    align = lambda x: (x + 255) // 256 * 256
    off_info = align(4 * 65)
    off_ml = align(off_info + 16 * cap)
    off_o = align(off_ml + 8 * cap * 16)
    total = align(off_o + 4 * cap * 16 * 128)
    assert lib.pkv_paged_decode_workspace_bytes(64, 16, 4096, CacheDesc(572, 256, 8, 128)) == total


def test_host_checks_return_codes_without_a_gpu(lib):
    from paged_kv_attention_scatter_gb300._binding import CacheDesc
    c = CacheDesc(8, 4, 1, 64)
    # empty calls are no-ops that launch nothing
    assert lib.pkv_kv_store(None, None, None, None, None, 0, c, None, None) == 0
    assert lib.pkv_sample(None, None, None, 0, 10, None, None, None) == 0
    # argument errors are reported before any CUDA call
    assert lib.pkv_kv_store(None, None, None, None, None, 3, c, None, None) == -1
    assert lib.pkv_kv_store(None, None, None, None, None, -1, c, None, None) == -2
    bad = CacheDesc(8, 4, 1, 96)
    assert lib.pkv_paged_decode(None, None, None, None, 1, None, 1, 1, 8, 1.0, None, None, 0,
                                bad, None, None) == -3
    assert lib.pkv_paged_decode(None, None, None, None, 1, None, 1, 3, 8, 1.0, None, None, 0,
                                CacheDesc(8, 4, 2, 64), None, None) == -2
    assert lib.pkv_paged_prefill_varlen(None, None, None, None, None, None, None, 1, 4, 4, 4,
                                        2, None, 0, 1.0, None, None, 0, c, None, None) == -1
    # the fused store + prefill checks the prefill's arguments before enqueueing the store
    assert lib.pkv_kv_store_paged_prefill_varlen(None, None, None, None, None, None, None, None,
                                                 1, 4, 4, 4, 2, None, 0, 1.0, None, None, 0, c,
                                                 None, None) == -1
    assert lib.pkv_kv_store_paged_prefill_varlen(None, None, None, None, None, None, None, None,
                                                 1, 4, 4, 4, 2, None, 0, 0.0, None, None, 0, c,
                                                 None, None) == -2
    # the decode plan checks what it depends on
    assert lib.pkv_paged_decode_plan(None, 2, 2, 8, 2, None, 0, c, None, None) == -1
    assert lib.pkv_paged_decode_plan(None, 2, 2, 8, 2, None, 0, bad, None, None) == -3
    assert lib.pkv_paged_decode_plan(None, 0, 2, 8, 2, None, 0, c, None, None) == 0
    assert lib.pkv_paged_decode_run(None, None, None, None, 2, None, 2, 2, 8, 1.0, None, None,
                                    0, c, None, None) == -1
    # a misaligned pointer is rejected on the host; it is never dereferenced
    p = ctypes.c_void_p(16 * 1024 + 2)
    assert lib.pkv_paged_decode_plan(p, 2, 2, 8, 2, p, 1 << 20, c, None, None) == -4
    assert lib.pkv_sample(p, p, p, 1, 10, p, None, None) == -4
    assert lib.pkv_kv_store_paged_prefill_varlen(p, p, p, p, p, p, p, p, 1, 4, 4, 4, 2, None, 0,
                                                 1.0, p, p, 1 << 20, c, None, None) == -4
    # the mixed-batch call: the prefill's checks, then block tables and the
    # combined workspace, all before anything is enqueued
    mixed = lib.pkv_kv_store_paged_attention_varlen
    assert mixed(None, None, None, None, None, None, None, None, 1, 4, 4, 4, 2, None, 0, 1.0,
                 None, None, 0, c, None, None) == -1
    ok = ctypes.c_void_p(16 * 1024)
    assert mixed(ok, ok, ok, ok, ok, ok, ok, ok, 1, 4, 4, 4, 2, None, 0, 1.0, ok, ok, 1 << 20,
                 c, None, None) == -1
    pre = lib.pkv_paged_prefill_workspace_bytes(1, 4, 2, c)
    assert mixed(ok, ok, ok, ok, ok, ok, ok, ok, 1, 4, 4, 4, 2, ok, 1, 1.0, ok, ok, pre, c,
                 None, None) == -5
    assert mixed(ok, ok, ok, ok, ok, ok, ok, ok, 1, 4, 4, 4, 2, ok, 1, 1.0, ok, p, 1 << 20, c,
                 None, None) == -4


def test_layer_cache_pointer_arithmetic(lib):
    """[LIFE] §2.2.3: the pool is [2, L, NB, bs, Hkv, D]; layer l's K is
    kv_cache[0, l] and its V kv_cache[1, l] (views).  Host arithmetic only."""
    from paged_kv_attention_scatter_gb300._binding import CacheDesc
    c = CacheDesc(10, 16, 2, 64)
    layer_bytes = 10 * 16 * 2 * 64 * 2
    base = 1 << 20
    kp, vp = ctypes.c_void_p(), ctypes.c_void_p()
    assert lib.pkv_layer_cache(base, 4, 3, c, ctypes.byref(kp), ctypes.byref(vp)) == 0
    assert kp.value == base + 3 * layer_bytes
    assert vp.value == base + (4 + 3) * layer_bytes
    assert lib.pkv_layer_cache(base, 4, 4, c, ctypes.byref(kp), ctypes.byref(vp)) == -2
    assert lib.pkv_layer_cache(None, 4, 0, c, ctypes.byref(kp), ctypes.byref(vp)) == -1


def test_mixed_batch_binding_checks_before_the_library(lib):
    """The Python binding of the mixed-batch call rejects a slot list of the
    wrong length and a missing block table before touching the library."""
    import pytest
    import torch
    from paged_kv_attention_scatter_gb300 import _binding
    q = torch.zeros(5, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(5, 1, 64, dtype=torch.bfloat16)
    cache = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 1, 5], dtype=torch.int32)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="one slot per query token"):
        _binding.kv_store_paged_attention_varlen(q, k, k, cache, cache,
                                                 torch.zeros(4, dtype=torch.int32), cu, cu,
                                                 4, 4, bt, 0.125)
    with pytest.raises(ValueError, match="block_tables is required"):
        _binding.kv_store_paged_attention_varlen(q, k, k, cache, cache,
                                                 torch.zeros(5, dtype=torch.int32), cu, cu,
                                                 4, 4, None, 0.125)
