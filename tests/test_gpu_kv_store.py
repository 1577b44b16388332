"""kv_store on the GPU against the oracle: bit-exact caches."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import kv_store as okv
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(pkv, k, v, kc, vc, slots, dev):
    st = pkv.new_status(dev)
    kd, vd = kc.to(dev), vc.to(dev)
    pkv.kv_store(k.to(dev), v.to(dev), kd, vd, slots.to(dev), status=st)
    ok, ov, bad = okv.kv_store(U.bits(k), U.bits(v), U.bits(kc), U.bits(vc), slots.numpy())
    assert np.array_equal(U.bits(kd), ok) and np.array_equal(U.bits(vd), ov)
    return U.status_word(st), bad


def test_tiny_prefill_and_decode_slots(cuda):
    pkv = U.lib()
    w = W.tiny_workload()
    p = w.prefill
    word, _ = _run(pkv, p.k, p.v, w.k_cache0, w.v_cache0, p.slot_mapping, cuda)
    assert word == 0
    st = w.decode_steps[1]                   # the step that crosses into a new block
    word, _ = _run(pkv, st.k_new, st.v_new, w.k_cache0, w.v_cache0, st.slot_mapping, cuda)
    assert word == 0


def test_prefill_chunk_rows_2kib(cuda):
    pkv = U.lib()
    spec = W.PrefillSpec("kv", seed=11, num_prompts=6, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, block_size=256, len_lo=300, len_hi=2000,
                         max_cached_blocks=2, token_budget=4096)
    w = W.prefill_workload(spec)
    st = w.steps[0]
    word, _ = _run(pkv, st.k, st.v, w.k_cache0, w.v_cache0, st.slot_mapping, cuda)
    assert word == 0


def test_decode_step_new_tokens(cuda):
    pkv = U.lib()
    spec = W.DecodeSpec("kv-step", seed=4, batch=512, num_q_heads=32, num_kv_heads=8,
                        head_dim=128, block_size=256, ctx_lo=256, ctx_hi=2048,
                        store_new_token=True)
    w = W.decode_workload(spec)
    word, _ = _run(pkv, w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, cuda)
    assert word == 0


def test_padding_and_out_of_range_slots(cuda):
    pkv = U.lib()
    g = torch.Generator().manual_seed(3)
    nb, bs, hkv, d = 6, 4, 2, 64
    kc = U.bf16_case(g, (nb, bs, hkv, d))
    vc = U.bf16_case(g, (nb, bs, hkv, d))
    k = U.bf16_case(g, (5, hkv, d))
    v = U.bf16_case(g, (5, hkv, d))
    slots = torch.tensor([3, -1, nb * bs, 23, -7], dtype=torch.int32)
    word, bad = _run(pkv, k, v, kc, vc, slots, cuda)
    assert bad == [nb * bs]
    assert word == pkv.STATUS["SLOT_OUT_OF_RANGE"]


def test_empty_call_is_a_noop(cuda):
    pkv = U.lib()
    kc = torch.zeros((2, 4, 1, 64), dtype=torch.bfloat16, device=cuda)
    e = torch.zeros((0, 1, 64), dtype=torch.bfloat16, device=cuda)
    pkv.kv_store(e, e, kc, kc.clone(), torch.zeros(0, dtype=torch.int32, device=cuda))
    assert int(kc.abs().sum()) == 0
