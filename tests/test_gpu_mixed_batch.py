"""Mixed prefill/decode batches: one call over a varlen batch whose sequences
are prefill chunks (several new tokens) and decode rows (one new token).

The pages' scheduler runs a step as all prefill or all decode ("一个 prompt 的一
生" §3.2), but a decode row is a chunk of one token (§3.1), so continuous
batching can take both together.  pkv_kv_store_paged_attention_varlen stores
the step's rows, runs the multi-query sequences through the varlen prefill
kernels and the one-query sequences through the split-KV decode kernels.
Checked here: the float64 oracle on every row; the multi-query rows equal to
kv_store_paged_prefill_varlen's and the one-query rows equal to paged_decode's
(same kernels, same chunking); degenerate batches (all decode, all prefill);
inconsistent one-query rows reported and left unwritten; replay from a CUDA
graph."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from test_gpu_fused_prefill import _same, _slots
from test_gpu_prefill import make_case

pytestmark = pytest.mark.gpu

# (Hq, Hkv, D, block size): TMA decode + tcgen05 prefill reading cached tiles
# as TMA boxes; register decode + tcgen05 prefill with per-block boxes and
# gathered V rows (16) or all rows gathered with cp.async (48); head_dim 64
# with TMA decode and per-block prefill boxes (64)
SHAPES = [(8, 2, 128, 256), (8, 2, 128, 16), (4, 1, 64, 64), (6, 3, 128, 48)]


def _run_case(pkv, dev, c, lens, cached, bs, scale, status=None, out=None):
    sl = _slots(c, lens, cached, bs).to(dev)
    q, k, v = c["q"].to(dev), c["k"].to(dev), c["v"].to(dev)
    cu_q, cu_k, bt = c["cu_q"].to(dev), c["cu_k"].to(dev), c["bt"].to(dev)
    kc, vc = c["kc"].to(dev), c["vc"].to(dev)
    o = pkv.kv_store_paged_attention_varlen(q, k, v, kc, vc, sl, cu_q, cu_k, c["max_sq"],
                                            c["max_sk"], bt, scale, out=out, status=status)
    return o, kc, vc, sl


def _decode_rows(pkv, dev, c, kc, vc, scale):
    """paged_decode over the same batch (every sequence, its last query row,
    all its keys from the cache): the decode pass's own chunking."""
    cu_q, cu_k = c["cu_q"].numpy(), c["cu_k"].numpy()
    B = len(cu_q) - 1
    last = torch.tensor([max(int(cu_q[b + 1]) - 1, 0) for b in range(B)], dtype=torch.long)
    q_last = c["q"][last].to(dev)
    ctx = torch.tensor(np.diff(cu_k), dtype=torch.int32, device=dev)
    return pkv.paged_decode(q_last, kc, vc, c["bt"].to(dev), ctx, scale, c["max_sk"])


@pytest.mark.parametrize("hq,hkv,d,bs", SHAPES)
def test_mixed_batch_matches_oracle_and_both_paths(cuda, hq, hkv, d, bs):
    pkv = U.lib()
    lens = [1, 300, 1, 1, 129, 1, 64, 1]
    cached = [700, 0, 2 * bs + 5, 0, bs, 1234, 17, bs - 1]
    c = make_case(311 + d + bs, lens, cached, hq, hkv, d, bs)
    scale = d ** -0.5
    st = pkv.new_status(cuda)
    o, kc, vc, sl = _run_case(pkv, cuda, c, lens, cached, bs, scale, status=st)
    # the reference paths on a fresh copy of the cache
    kc2, vc2 = c["kc"].to(cuda), c["vc"].to(cuda)
    o_pre = pkv.kv_store_paged_prefill_varlen(c["q"].to(cuda), c["k"].to(cuda), c["v"].to(cuda),
                                              kc2, vc2, sl, c["cu_q"].to(cuda),
                                              c["cu_k"].to(cuda), c["max_sq"], c["max_sk"],
                                              c["bt"].to(cuda), scale)
    o_dec = _decode_rows(pkv, cuda, c, kc2, vc2, scale)
    torch.cuda.synchronize()
    assert U.status_word(st) == 0
    assert _same(kc, kc2) and _same(vc, vc2)
    cu_q = c["cu_q"].numpy()
    for b, n in enumerate(lens):
        rows = slice(int(cu_q[b]), int(cu_q[b + 1]))
        if n == 1:
            assert torch.equal(o[rows], o_dec[b:b + 1]), f"decode row {b}"
        else:
            assert torch.equal(o[rows], o_pre[rows]), f"prefill rows of sequence {b}"
    ref = oatt.paged_prefill_varlen(U.f64(c["q"]), U.f64(c["k"]), U.f64(c["v"]), c["kc"],
                                    c["vc"], cu_q, c["cu_k"].numpy(), c["bt"].numpy(), scale)
    U.assert_close(U.f64(o), ref, "mixed batch")


@pytest.mark.parametrize("hq,hkv,d,bs", [(8, 2, 128, 256), (6, 3, 128, 48)])
def test_all_decode_rows_and_all_prefill_rows(cuda, hq, hkv, d, bs):
    """An empty prefill schedule and an empty decode plan are both fine."""
    pkv = U.lib()
    scale = d ** -0.5
    for seed, lens, cached in ((5, [1] * 37, [(i * 97) % 900 for i in range(37)]),
                               (6, [3, 130, 2, 64], [bs, 0, 77, 2 * bs])):
        c = make_case(seed + d, lens, cached, hq, hkv, d, bs)
        st = pkv.new_status(cuda)
        o, _, _, _ = _run_case(pkv, cuda, c, lens, cached, bs, scale, status=st)
        torch.cuda.synchronize()
        assert U.status_word(st) == 0
        ref = oatt.paged_prefill_varlen(U.f64(c["q"]), U.f64(c["k"]), U.f64(c["v"]), c["kc"],
                                        c["vc"], c["cu_q"].numpy(), c["cu_k"].numpy(),
                                        c["bt"].numpy(), scale)
        U.assert_close(U.f64(o), ref, f"lens {lens[:4]}")


def test_inconsistent_decode_row_is_reported_and_not_written(cuda):
    """A one-query sequence with more keys than max_seqlen_k is rejected by the
    decode plan (its chunk plan is sized by max_seqlen_k): the status word
    says so, its output row keeps its old contents, the other rows are right."""
    pkv = U.lib()
    hq, hkv, d, bs = 8, 2, 128, 256
    lens, cached = [1, 40, 1], [300, 10, 600]
    c = make_case(77, lens, cached, hq, hkv, d, bs)
    scale = d ** -0.5
    c_bad = dict(c)
    c_bad["max_sk"] = 400                  # sequence 2 has 601 keys
    out = torch.full_like(c["q"], 3.0).to(cuda)
    st = pkv.new_status(cuda)
    o, _, _, _ = _run_case(pkv, cuda, c_bad, lens, cached, bs, scale, status=st, out=out)
    torch.cuda.synchronize()
    word = U.status_word(st)
    assert word & pkv.STATUS["BAD_SEQLENS"]
    assert torch.all(o[41] == 3.0)
    ref = oatt.paged_prefill_varlen(U.f64(c["q"]), U.f64(c["k"]), U.f64(c["v"]), c["kc"],
                                    c["vc"], c["cu_q"].numpy(), c["cu_k"].numpy(),
                                    c["bt"].numpy(), scale)
    U.assert_close(U.f64(o[:41]), ref[:41], "rows of the consistent sequences")


def test_mixed_batch_in_a_cuda_graph(cuda):
    pkv = U.lib()
    hq, hkv, d, bs = 8, 2, 128, 256
    lens = [1, 200, 1, 1, 77]
    cached = [500, bs, 3, 1000, 0]
    c = make_case(404, lens, cached, hq, hkv, d, bs)
    scale = d ** -0.5
    sl = _slots(c, lens, cached, bs).to(cuda)
    q, k, v = c["q"].to(cuda), c["k"].to(cuda), c["v"].to(cuda)
    cu_q, cu_k, bt = c["cu_q"].to(cuda), c["cu_k"].to(cuda), c["bt"].to(cuda)
    kc0, vc0 = c["kc"].to(cuda), c["vc"].to(cuda)
    kc1, vc1 = kc0.clone(), vc0.clone()
    o1 = pkv.kv_store_paged_attention_varlen(q, k, v, kc1, vc1, sl, cu_q, cu_k, c["max_sq"],
                                             c["max_sk"], bt, scale)
    kc2, vc2 = kc0.clone(), vc0.clone()
    out = torch.empty_like(q)
    ws = torch.empty(pkv.paged_attention_varlen_workspace_bytes(len(lens), q.shape[0], hq,
                                                                c["max_sk"], kc2.shape),
                     dtype=torch.uint8, device=cuda)
    st = pkv.new_status(cuda)

    def call():
        pkv.kv_store_paged_attention_varlen(q, k, v, kc2, vc2, sl, cu_q, cu_k, c["max_sq"],
                                            c["max_sk"], bt, scale, out=out, workspace=ws,
                                            status=st)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                   # warm-up outside the capture
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    kc2.copy_(kc0)
    vc2.copy_(vc0)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert U.status_word(st) == 0
    assert _same(kc1, kc2) and _same(vc1, vc2)
    assert torch.equal(o1, out)


def test_mixed_8b_sampled_rows(cuda):
    """The benchmark's mixed-8b step (256 decode rows and 4 prefill chunks,
    32/8 heads, 256-slot blocks) in the call bench.py times; the oracle
    computes sampled rows one by one: 32 decode rows and 8 rows of each chunk."""
    pkv = U.lib()
    from paged_kv_attention_scatter_gb300 import workloads as W
    spec = W.MIXED_8B
    w = W.mixed_workload(spec, device=cuda)
    st = w.step
    kc0, vc0 = w.k_cache0.cpu(), w.v_cache0.cpu()          # before the store
    status = pkv.new_status(cuda)
    out = pkv.kv_store_paged_attention_varlen(
        st.q, st.k, st.v, w.k_cache0, w.v_cache0, st.slot_mapping.to(cuda),
        st.cu_seqlens_q.to(cuda), st.cu_seqlens_k.to(cuda), st.max_seqlen_q, st.max_seqlen_k,
        st.block_tables.to(cuda), w.scale, status=status)
    assert U.status_word(status) == 0
    cu_q = st.cu_seqlens_q.numpy()
    rng = np.random.default_rng(5)
    rows = {int(b): [0] for b in rng.choice(spec.num_decode, size=32, replace=False)}
    for b in range(spec.num_decode, spec.num_decode + spec.num_prefill):
        n = int(cu_q[b + 1] - cu_q[b])
        rows[b] = sorted({0, n - 1} | set(rng.integers(0, n, size=6).tolist()))
    ref = oatt.paged_prefill_varlen(U.f64(st.q.cpu()), U.f64(st.k.cpu()), U.f64(st.v.cpu()),
                                    kc0, vc0, cu_q, st.cu_seqlens_k.numpy(),
                                    st.block_tables.numpy(), w.scale, rows=rows)
    mask = ~np.isnan(ref[:, 0, 0])
    assert mask.sum() == 32 + sum(len(r) for b, r in rows.items() if b >= spec.num_decode)
    err, rel = U.assert_close(U.f64(out)[mask], ref[mask], "mixed-8b sampled rows")
    print(f"mixed-8b: {mask.sum()} rows, max abs {err:.3g}, rel L2 {rel:.3g}")
