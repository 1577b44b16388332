"""The fused store-then-decode entry point and the multi-layer pool view.

* pkv_kv_store_paged_decode must give exactly what pkv_kv_store followed by
  pkv_paged_decode gives (same kernels, chained launches), also when captured
  in CUDA graphs for each batch size of the pages' ladder
  ("一个 prompt 的一生" §2.2.4: graph_bs = [1, 2, 4, 8] + range(16, max_bs+1, 16)).
* Decoding through layer_cache views of a [2, L, NB, bs, Hkv, D] pool equals
  decoding the same layer held in separate tensors."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from oracle import kv_store as okv
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SPEC = W.DecodeSpec("ladder", seed=23, batch=48, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    block_size=256, ctx_lo=50, ctx_hi=2500, store_new_token=True)


def test_fused_equals_separate_calls(cuda):
    pkv = U.lib()
    w = W.decode_workload(SPEC, device=cuda)
    bt, ctx, sl = w.block_tables.to(cuda), w.context_lens.to(cuda), w.slot_mapping.to(cuda)
    kc1, vc1 = w.k_cache.clone(), w.v_cache.clone()
    kc2, vc2 = w.k_cache.clone(), w.v_cache.clone()
    pkv.kv_store(w.k_new, w.v_new, kc1, vc1, sl)
    o1 = pkv.paged_decode(w.q, kc1, vc1, bt, ctx, w.scale, w.max_context_len)
    st = pkv.new_status(cuda)
    o2 = pkv.kv_store_paged_decode(w.k_new, w.v_new, sl, w.q, kc2, vc2, bt, ctx, w.scale,
                                   w.max_context_len, status=st)
    assert U.status_word(st) == 0
    assert torch.equal(kc1, kc2) or (torch.isnan(kc1) == torch.isnan(kc2)).all() and \
        torch.equal(torch.nan_to_num(kc1), torch.nan_to_num(kc2))
    assert torch.equal(o1, o2)


def test_fused_step_graph_per_ladder_batch_size(cuda):
    pkv = U.lib()
    w = W.decode_workload(SPEC)                 # CPU copy for the oracle
    ladder = [1, 2, 4, 8] + list(range(16, SPEC.batch + 1, 16))
    kc, vc = w.k_cache.to(cuda), w.v_cache.to(cuda)
    # static buffers at the largest batch; a graph of batch n uses the first n rows
    q, kn, vn = w.q.to(cuda), w.k_new.to(cuda), w.v_new.to(cuda)
    sl, bt, ctx = w.slot_mapping.to(cuda), w.block_tables.to(cuda), w.context_lens.to(cuda)
    out = torch.zeros_like(q)
    # one workspace serves every graph: size it for the largest requirement
    need = max(pkv.paged_decode_workspace_bytes(n, 32, SPEC.ctx_hi, kc) for n in ladder)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda)
    graphs = {}
    for n in reversed(ladder):                  # largest first, as the pages capture
        fn = lambda n=n: pkv.kv_store_paged_decode(kn[:n], vn[:n], sl[:n], q[:n], kc, vc,
                                                   bt[:n], ctx[:n], w.scale, SPEC.ctx_hi,
                                                   out=out[:n], workspace=ws)
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[n] = g
    okc, ovc, _ = okv.kv_store(U.bits(w.k_new), U.bits(w.v_new), U.bits(w.k_cache),
                               U.bits(w.v_cache), w.slot_mapping.numpy())
    kt = torch.from_numpy(okc).view(torch.bfloat16)
    vt = torch.from_numpy(ovc).view(torch.bfloat16)
    ref = oatt.paged_decode(U.f64(w.q), kt, vt, w.block_tables.numpy(), w.context_lens.numpy(),
                            w.scale)
    for n in ladder:
        out.zero_()
        graphs[n].replay()
        torch.cuda.synchronize()
        got = U.f64(out)
        U.assert_close(got[:n], ref[:n], f"ladder batch {n}")
        assert np.all(got[n:] == 0.0)


def test_decode_through_a_multi_layer_pool(cuda):
    pkv = U.lib()
    spec = W.DecodeSpec("pool", seed=29, batch=6, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        block_size=16, ctx_lo=20, ctx_hi=300)
    w = W.decode_workload(spec, device=cuda)
    L = 3
    pool = torch.zeros((2, L) + tuple(w.k_cache.shape), dtype=torch.bfloat16, device=cuda)
    pool[0, 2].copy_(w.k_cache)
    pool[1, 2].copy_(w.v_cache)
    kc, vc = pkv.layer_cache(pool, 2)
    bt, ctx = w.block_tables.to(cuda), w.context_lens.to(cuda)
    a = pkv.paged_decode(w.q, kc, vc, bt, ctx, w.scale, w.max_context_len)
    b = pkv.paged_decode(w.q, w.k_cache, w.v_cache, bt, ctx, w.scale, w.max_context_len)
    assert torch.equal(a, b)


@pytest.mark.parametrize("bs", [256, 16])
def test_plan_once_run_per_layer(cuda, bs):
    """pkv_paged_decode_plan once, then pkv_paged_decode_run for each layer of
    a [2, L, NB, bs, Hkv, D] pool: each layer's output is exactly what
    pkv_paged_decode gives, eagerly and replayed from one CUDA graph; a context
    length the plan rejects is reported and its rows are zero."""
    pkv = U.lib()
    spec = W.DecodeSpec("plan-run", seed=31, batch=20, num_q_heads=16, num_kv_heads=4,
                        head_dim=128, block_size=bs, ctx_lo=1, ctx_hi=1500)
    w = W.decode_workload(spec, device=cuda)
    L = 3
    g = torch.Generator().manual_seed(5)
    pool = torch.empty((2, L) + tuple(w.k_cache.shape), dtype=torch.bfloat16, device=cuda)
    for layer in range(L):
        pool[0, layer].copy_(torch.randn(w.k_cache.shape, generator=g).to(torch.bfloat16))
        pool[1, layer].copy_(torch.randn(w.v_cache.shape, generator=g).to(torch.bfloat16))
    layers = [pkv.layer_cache(pool, layer) for layer in range(L)]
    bt, ctx = w.block_tables.to(cuda), w.context_lens.to(cuda)
    max_ctx = w.max_context_len
    refs = [pkv.paged_decode(w.q, kc, vc, bt, ctx, w.scale, max_ctx) for kc, vc in layers]
    st = pkv.new_status(cuda)
    ws = pkv.paged_decode_plan(ctx, spec.num_q_heads, max_ctx, bt.shape[1], layers[0][0],
                               status=st)
    outs = [pkv.paged_decode_run(w.q, kc, vc, bt, ctx, w.scale, max_ctx, ws, status=st)
            for kc, vc in layers]
    torch.cuda.synchronize()
    assert U.status_word(st) == 0
    for o, r in zip(outs, refs):
        assert torch.equal(o, r)
    # the same step captured in one graph
    outs_g = [torch.empty_like(w.q) for _ in layers]

    def step():
        pkv.paged_decode_plan(ctx, spec.num_q_heads, max_ctx, bt.shape[1], layers[0][0],
                              workspace=ws, status=st)
        for (kc, vc), o in zip(layers, outs_g):
            pkv.paged_decode_run(w.q, kc, vc, bt, ctx, w.scale, max_ctx, ws, out=o, status=st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for o in outs_g:
        o.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for o, r in zip(outs_g, refs):
        assert torch.equal(o, r)
    # a rejected context length: reported by the plan, zero rows from the run
    bad = ctx.clone()
    bad[3] = max_ctx + 1
    st2 = pkv.new_status(cuda)
    ws2 = pkv.paged_decode_plan(bad, spec.num_q_heads, max_ctx, bt.shape[1], layers[0][0],
                                status=st2)
    o2 = pkv.paged_decode_run(w.q, layers[0][0], layers[0][1], bt, bad, w.scale, max_ctx, ws2)
    torch.cuda.synchronize()
    assert U.status_word(st2) == pkv.STATUS["BAD_CONTEXT_LEN"]
    assert float(o2[3].abs().max()) == 0.0
    keep = [b for b in range(spec.batch) if b != 3]
    assert torch.equal(o2[keep], refs[0][keep])
