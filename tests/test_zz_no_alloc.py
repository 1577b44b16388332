"""pkv_paged_decode_static_workspace: decode for callers that cannot allocate
device memory where they call (a plugin whose host engine owns all device
memory, a loop that must not pay for cudaMalloc's implicit synchronisation).

Its scratch is a fixed array inside the library.  This file is collected last
so that, if it fails, a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process."""
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from paged_kv_attention_scatter_gb300 import _binding
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(spec, dev):
    w = W.decode_workload(spec, device=dev)
    return w, w.block_tables.to(dev), w.context_lens.to(dev)


def _compare_with_workspace_entry_point(pkv, w, bt, ctx, dev):
    """The static-workspace call against pkv_paged_decode (same kernels, so
    bit for bit) and against the float64 oracle (within the attention
    tolerance)."""
    ref = pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len)
    st = pkv.new_status(dev)
    got = _binding.paged_decode_static_workspace(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale,
                                                 w.max_context_len, status=st)
    assert U.status_word(st) == 0
    U.assert_close(U.f64(got), U.f64(ref), "static-workspace decode vs workspace decode")
    assert torch.equal(got, ref)
    oracle = oatt.paged_decode(U.f64(w.q), w.k_cache.cpu(), w.v_cache.cpu(),
                               w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    U.assert_close(U.f64(got), oracle, "static-workspace decode vs the oracle")


def test_two_calls_in_a_row_match_the_workspace_entry_point(cuda):
    pkv = U.lib()
    # decode-0.6b needs about 8.5 MB of scratch; a second, different call must
    # not see anything left over from the first
    w1, bt1, ctx1 = _inputs(W.DECODE_0P6B, cuda)
    need = pkv.paged_decode_workspace_bytes(64, 16, w1.max_context_len, w1.k_cache)
    assert need <= _binding.STATIC_DECODE_WORKSPACE_BYTES
    _compare_with_workspace_entry_point(pkv, w1, bt1, ctx1, cuda)
    spec2 = W.DecodeSpec("second call", seed=77, batch=37, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, block_size=16, ctx_lo=1, ctx_hi=1500)
    w2, bt2, ctx2 = _inputs(spec2, cuda)
    _compare_with_workspace_entry_point(pkv, w2, bt2, ctx2, cuda)


def test_sizes_beyond_the_array_are_rejected(cuda):
    pkv = U.lib()
    # 256 sequences of up to 32768 keys, 64 q heads: far more scratch than the array
    kc_shape = torch.zeros((1, 256, 8, 128), dtype=torch.bfloat16)
    assert pkv.paged_decode_workspace_bytes(256, 64, 32768, kc_shape) > \
        _binding.STATIC_DECODE_WORKSPACE_BYTES
    q = torch.zeros((256, 64, 128), dtype=torch.bfloat16, device=cuda)
    kc = torch.zeros((1, 256, 8, 128), dtype=torch.bfloat16, device=cuda)
    bt = torch.zeros((256, 128), dtype=torch.int32, device=cuda)
    ctx = torch.zeros(256, dtype=torch.int32, device=cuda)
    with pytest.raises(RuntimeError, match="workspace"):
        _binding.paged_decode_static_workspace(q, kc, kc, bt, ctx, 0.1, 32768)
