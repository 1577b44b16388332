"""The fused store-then-prefill entry point (a prefill round's per-layer pair,
"一个 prompt 的一生" §2.2.4 and §4: store_kvcache, then the attention op).

pkv_kv_store_paged_prefill_varlen must leave the cache exactly as pkv_kv_store
leaves it and give exactly the output of pkv_paged_prefill_varlen (same
kernels, chained launches), with every way the tcgen05 kernel loads cached
tiles (TMA boxes for block sizes that are multiples of 128; per-block boxes
for K and most of V with the rest of V gathered with cp.async at 16, 32, 8;
rows gathered for both at 4, 48), eagerly and replayed from a CUDA graph; its
output also matches the float64 oracle."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from test_gpu_prefill import make_case

pytestmark = pytest.mark.gpu

SHAPES = [(8, 2, 128, 256), (8, 2, 128, 128), (4, 1, 64, 16), (6, 3, 128, 32), (4, 2, 128, 4),
          (8, 2, 64, 48), (4, 2, 128, 8)]


def _slots(c, lens, cached, bs):
    """Slot of every new token: block_tables[b][p // bs] * bs + p % bs for
    positions p = cached[b] .. cached[b] + lens[b] - 1, with padding (-1) rows
    where a sequence has no new token."""
    bt = c["bt"]
    out = []
    for b, (n, cb) in enumerate(zip(lens, cached)):
        for p in range(cb, cb + n):
            out.append(int(bt[b, p // bs]) * bs + p % bs)
    return torch.tensor(out, dtype=torch.int32)


def _same(a, b):
    return torch.equal(torch.nan_to_num(a, nan=7.0), torch.nan_to_num(b, nan=7.0)) and \
        torch.equal(torch.isnan(a), torch.isnan(b))


@pytest.mark.parametrize("hq,hkv,d,bs", SHAPES)
def test_fused_prefill_equals_store_then_prefill(cuda, hq, hkv, d, bs):
    pkv = U.lib()
    lens = [300, 1, 129, 64, 200]
    cached = [0, 2 * bs + 5, bs, 17, 3]
    c = make_case(41 + d + bs, lens, cached, hq, hkv, d, bs)
    sl = _slots(c, lens, cached, bs).to(cuda)
    q, k, v = c["q"].to(cuda), c["k"].to(cuda), c["v"].to(cuda)
    cu_q, cu_k, bt = c["cu_q"].to(cuda), c["cu_k"].to(cuda), c["bt"].to(cuda)
    scale = d ** -0.5
    kc1, vc1 = c["kc"].to(cuda), c["vc"].to(cuda)
    kc2, vc2 = kc1.clone(), vc1.clone()
    pkv.kv_store(k, v, kc1, vc1, sl)
    o1 = pkv.paged_prefill_varlen(q, k, v, kc1, vc1, cu_q, cu_k, c["max_sq"], c["max_sk"], bt,
                                  scale)
    st = pkv.new_status(cuda)
    o2 = pkv.kv_store_paged_prefill_varlen(q, k, v, kc2, vc2, sl, cu_q, cu_k, c["max_sq"],
                                           c["max_sk"], bt, scale, status=st)
    torch.cuda.synchronize()
    assert U.status_word(st) == 0
    assert _same(kc1, kc2) and _same(vc1, vc2)
    assert torch.equal(o1, o2)
    ref = oatt.paged_prefill_varlen(U.f64(c["q"]), U.f64(c["k"]), U.f64(c["v"]), c["kc"],
                                    c["vc"], c["cu_q"].numpy(), c["cu_k"].numpy(),
                                    c["bt"].numpy(), scale)
    U.assert_close(U.f64(o2), ref, "fused prefill")
    # the stored rows are this call's k/v rows at their slots
    flat_k = kc2.reshape(-1, hkv, d)
    assert torch.equal(flat_k[sl.long()], k)


@pytest.mark.parametrize("hq,hkv,d,bs", [(8, 2, 128, 256), (4, 1, 64, 16), (4, 2, 128, 48)])
def test_fused_prefill_in_a_cuda_graph(cuda, hq, hkv, d, bs):
    pkv = U.lib()
    lens = [128, 77, 1, 256]
    cached = [bs, 0, 3, 40]
    c = make_case(97 + d, lens, cached, hq, hkv, d, bs)
    sl = _slots(c, lens, cached, bs).to(cuda)
    q, k, v = c["q"].to(cuda), c["k"].to(cuda), c["v"].to(cuda)
    cu_q, cu_k, bt = c["cu_q"].to(cuda), c["cu_k"].to(cuda), c["bt"].to(cuda)
    scale = d ** -0.5
    kc0, vc0 = c["kc"].to(cuda), c["vc"].to(cuda)
    kc1, vc1 = kc0.clone(), vc0.clone()
    pkv.kv_store(k, v, kc1, vc1, sl)
    o1 = pkv.paged_prefill_varlen(q, k, v, kc1, vc1, cu_q, cu_k, c["max_sq"], c["max_sk"], bt,
                                  scale)
    kc2, vc2 = kc0.clone(), vc0.clone()
    out = torch.empty_like(q)
    ws = torch.empty(pkv.paged_prefill_workspace_bytes(len(lens), q.shape[0], hq, kc2.shape),
                     dtype=torch.uint8, device=cuda)
    st = pkv.new_status(cuda)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                   # warm-up outside the capture
        pkv.kv_store_paged_prefill_varlen(q, k, v, kc2, vc2, sl, cu_q, cu_k, c["max_sq"],
                                          c["max_sk"], bt, scale, out=out, workspace=ws,
                                          status=st)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.kv_store_paged_prefill_varlen(q, k, v, kc2, vc2, sl, cu_q, cu_k, c["max_sq"],
                                          c["max_sk"], bt, scale, out=out, workspace=ws,
                                          status=st)
    kc2.copy_(kc0)
    vc2.copy_(vc0)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert U.status_word(st) == 0
    assert _same(kc1, kc2) and _same(vc1, vc2)
    assert torch.equal(o1, out)
