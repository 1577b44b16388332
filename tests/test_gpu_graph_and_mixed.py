"""The hot path inside a CUDA graph, and decode rows inside a varlen prefill.

* The pages' decode step is replayed from a CUDA graph with static input
  buffers whose contents change between replays ("一个 prompt 的一生" §2.2.4:
  graph_vars are preallocated and refilled, then replayed).  The calls
  allocate nothing and never synchronise, so the whole step (kv_store,
  paged_decode, sample) is captured once and replayed on new data.
* Decode is prefill with one query per sequence: a single varlen prefill call
  over a batch that mixes one-query sequences with long chunks matches the
  oracle, and its one-query rows match paged_decode."""
import math

import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from oracle import kv_store as okv
from oracle import sampler as osm
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_decode_step_replayed_from_a_cuda_graph(cuda):
    pkv = U.lib()
    spec = W.DecodeSpec("graph", seed=31, batch=24, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=256, ctx_lo=100, ctx_hi=3000, store_new_token=True,
                        vocab=5000, logit_spikes=2, t_lo=0.3, t_hi=1.1)
    w0 = W.decode_workload(spec)
    # static buffers (graph_vars)
    kc, vc = w0.k_cache.to(cuda), w0.v_cache.to(cuda)
    st = {n: getattr(w0, n).to(cuda).clone() for n in
          ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens", "logits",
           "temperatures", "exp_noise")}
    out = torch.empty_like(st["q"])
    ids = torch.empty(spec.batch, dtype=torch.int32, device=cuda)
    ws = torch.empty(pkv.paged_decode_workspace_bytes(spec.batch, 32, 3000, kc),
                     dtype=torch.uint8, device=cuda)
    status = pkv.new_status(cuda)

    def step():
        pkv.kv_store(st["k_new"], st["v_new"], kc, vc, st["slot_mapping"], status=status)
        pkv.paged_decode(st["q"], kc, vc, st["block_tables"], st["context_lens"], w0.scale, 3000,
                         out=out, workspace=ws, status=status)
        pkv.sample(st["logits"], st["temperatures"], st["exp_noise"], out=ids, status=status)

    step()                                      # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    okc, ovc = U.bits(w0.k_cache), U.bits(w0.v_cache)
    g2 = torch.Generator().manual_seed(7)
    for replay in range(2):
        # new inputs for the same sequences: new query, new token K/V, new logits/noise
        q = U.bf16_case(g2, tuple(st["q"].shape))
        kn = U.bf16_case(g2, tuple(st["k_new"].shape))
        vn = U.bf16_case(g2, tuple(st["v_new"].shape))
        lg, tp, en = W.sampler_inputs(spec.batch, spec.vocab, 3.0, 2, 0.3, 1.1, g2)
        for name, t in (("q", q), ("k_new", kn), ("v_new", vn), ("logits", lg),
                        ("temperatures", tp), ("exp_noise", en)):
            st[name].copy_(t.to(cuda))
        g.replay()
        torch.cuda.synchronize()
        assert U.status_word(status) == 0
        okc, ovc, _ = okv.kv_store(U.bits(kn), U.bits(vn), okc, ovc, w0.slot_mapping.numpy())
        ref = oatt.paged_decode(U.f64(q), torch.from_numpy(okc).view(torch.bfloat16),
                                torch.from_numpy(ovc).view(torch.bfloat16),
                                w0.block_tables.numpy(), w0.context_lens.numpy(), w0.scale)
        U.assert_close(U.f64(out), ref, f"graph replay {replay}")
        ref_ids, _ = osm.sample(lg.numpy(), tp.numpy(), en.numpy())
        _, keys = osm.sample_key_form(lg.numpy(), tp.numpy(), en.numpy())
        near = osm.near_ties(keys)
        got = ids.cpu().numpy()
        for r in range(spec.batch):
            assert got[r] == ref_ids[r] or (len(near[r]) > 1 and got[r] in near[r])
    assert np.array_equal(U.bits(kc), okc)


@pytest.mark.parametrize("bs", [256, 16])
def test_one_query_sequences_inside_a_varlen_prefill(cuda, bs):
    pkv = U.lib()
    hq, hkv, d = 16, 4, 128
    lens = [1, 200, 1, 129, 1]
    cached = [300, 0, 1000, 2 * bs, 17]
    g = torch.Generator().manual_seed(41 + bs)
    K = [U.bf16_case(g, (c + n, hkv, d)) for n, c in zip(lens, cached)]
    V = [U.bf16_case(g, (c + n, hkv, d)) for n, c in zip(lens, cached)]
    q = U.bf16_case(g, (sum(lens), hq, d))
    nb = sum(-(-(c + n) // bs) for n, c in zip(lens, cached)) + 3
    kc, vc, bt = U.build_paged_cache(K, V, bs, nb, g)       # all keys already stored
    k = torch.cat([x[c:] for x, c in zip(K, cached)])
    v = torch.cat([x[c:] for x, c in zip(V, cached)])
    cu_q = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
    cu_k = torch.tensor([0] + np.cumsum([n + c for n, c in zip(lens, cached)]).tolist(),
                        dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    out = pkv.paged_prefill_varlen(q.to(cuda), k.to(cuda), v.to(cuda), kc.to(cuda), vc.to(cuda),
                                   cu_q.to(cuda), cu_k.to(cuda), max(lens),
                                   max(n + c for n, c in zip(lens, cached)), bt.to(cuda), scale)
    ref = oatt.paged_prefill_varlen(U.f64(q), U.f64(k), U.f64(v), kc, vc, cu_q.numpy(),
                                    cu_k.numpy(), bt.numpy(), scale)
    U.assert_close(U.f64(out), ref, "mixed varlen batch")
    # the one-query rows are exactly what paged_decode computes for those sequences
    rows = [int(cu_q[i]) for i, n in enumerate(lens) if n == 1]
    seqs = [i for i, n in enumerate(lens) if n == 1]
    ctx = torch.tensor([cached[i] + 1 for i in seqs], dtype=torch.int32)
    dec = pkv.paged_decode(q[rows].to(cuda).contiguous(), kc.to(cuda), vc.to(cuda),
                           bt[seqs].contiguous().to(cuda), ctx.to(cuda), scale, int(ctx.max()))
    U.assert_close(U.f64(dec), ref[rows], "decode rows")
