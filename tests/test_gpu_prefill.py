"""paged_prefill_varlen on the GPU against the float64 oracle."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from oracle import kv_store as okv
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _prefill(pkv, dev, q, k, v, kc, vc, cu_q, cu_k, bt, scale, max_sq, max_sk, status=None):
    return pkv.paged_prefill_varlen(q.to(dev), k.to(dev), v.to(dev),
                                    None if kc is None else kc.to(dev),
                                    None if vc is None else vc.to(dev),
                                    cu_q.to(dev), cu_k.to(dev), max_sq, max_sk,
                                    None if bt is None else bt.to(dev), scale, status=status)


def make_case(seed, lens, cached, hq, hkv, d, bs, spare=2):
    """Sequences with `cached[b]` tokens already in a paged cache and `lens[b]`
    new tokens in this call (bf16 values)."""
    g = torch.Generator().manual_seed(seed)
    K = [U.bf16_case(g, (c + n, hkv, d)) for n, c in zip(lens, cached)]
    V = [U.bf16_case(g, (c + n, hkv, d)) for n, c in zip(lens, cached)]
    q = U.bf16_case(g, (sum(lens), hq, d))
    nb = sum(-(-(c + n) // bs) for n, c in zip(lens, cached)) + spare
    kc, vc, bt = U.build_paged_cache([x[:c] for x, c in zip(K, cached)],
                                     [x[:c] for x, c in zip(V, cached)], bs, nb, g,
                                     extra_blocks_per_seq=[-(-(c + n) // bs)
                                                           for n, c in zip(lens, cached)])
    k = torch.cat([x[c:] for x, c in zip(K, cached)])
    v = torch.cat([x[c:] for x, c in zip(V, cached)])
    cu_q = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
    cu_k = torch.tensor([0] + np.cumsum([n + c for n, c in zip(lens, cached)]).tolist(),
                        dtype=torch.int32)
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, cu_q=cu_q, cu_k=cu_k, bt=bt,
                max_sq=max(lens), max_sk=max(n + c for n, c in zip(lens, cached)))


def _check_case(pkv, dev, c, scale, use_bt=True, rows=None):
    st = pkv.new_status(dev)
    out = _prefill(pkv, dev, c["q"], c["k"], c["v"], c["kc"] if use_bt else None,
                   c["vc"] if use_bt else None, c["cu_q"], c["cu_k"],
                   c["bt"] if use_bt else None, scale, c["max_sq"], c["max_sk"], status=st)
    assert U.status_word(st) == 0
    ref = oatt.paged_prefill_varlen(U.f64(c["q"]), U.f64(c["k"]), U.f64(c["v"]), c["kc"],
                                    c["vc"], c["cu_q"].numpy(), c["cu_k"].numpy(),
                                    c["bt"].numpy() if use_bt else None, scale, rows=rows)
    got = U.f64(out)
    mask = ~np.isnan(ref[:, 0, 0])
    return U.assert_close(got[mask], ref[mask], "prefill")


def test_tiny_with_and_without_block_tables(cuda):
    pkv = U.lib()
    w = W.tiny_workload()
    p = w.prefill
    outs = []
    for bt in (p.block_tables, None):
        out = _prefill(pkv, cuda, p.q, p.k, p.v, w.k_cache0, w.v_cache0, p.cu_seqlens_q,
                       p.cu_seqlens_k, bt, w.scale, p.max_seqlen_q, p.max_seqlen_k)
        ref = oatt.paged_prefill_varlen(U.f64(p.q), U.f64(p.k), U.f64(p.v), None, None,
                                        p.cu_seqlens_q.numpy(), p.cu_seqlens_k.numpy(), None,
                                        w.scale)
        U.assert_close(U.f64(out), ref, "tiny prefill")
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


# the tcgen05 kernel's ways of loading a cached 128-key tile: one TMA box per
# 64-column block (block sizes that are multiples of 128); K as one box per
# cache block and V the same for its first 64 rows (8, 64) or 96 rows (16, 32),
# the rest of V gathered with cp.async; or both gathered (4, 48, any other)
@pytest.mark.parametrize("hq,hkv,d,bs", [(8, 2, 128, 16), (4, 1, 64, 4), (6, 3, 128, 256),
                                         (2, 2, 64, 256), (16, 4, 128, 128), (8, 2, 128, 8),
                                         (4, 4, 128, 32), (8, 1, 128, 64), (4, 2, 128, 48),
                                         (4, 2, 64, 128), (8, 4, 64, 32), (6, 2, 64, 48),
                                         (4, 2, 64, 8), (8, 2, 64, 64), (2, 1, 64, 16)])
def test_ragged_cached_prefixes(cuda, hq, hkv, d, bs):
    pkv = U.lib()
    lens = [200, 1, 129, 64, 300]
    cached = [0, 48, 100, 17, 2 * bs]
    c = make_case(hq * 7 + d + bs, lens, cached, hq, hkv, d, bs)
    _check_case(pkv, cuda, c, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("d,bs", [(128, 256), (64, 256), (128, 16)])
def test_output_only_16_byte_aligned(cuda, d, bs):
    """An output buffer at a 16-byte (not 32-byte) boundary takes the 16-byte
    store path of the epilogue; its rows equal those of an aligned output."""
    pkv = U.lib()
    lens, cached = [200, 1, 129], [0, 48, 2 * bs]
    c = make_case(123 + d + bs, lens, cached, 8, 2, d, bs)
    args = (c["q"].to(cuda), c["k"].to(cuda), c["v"].to(cuda), c["kc"].to(cuda),
            c["vc"].to(cuda), c["cu_q"].to(cuda), c["cu_k"].to(cuda), c["max_sq"], c["max_sk"],
            c["bt"].to(cuda), 1.0 / math.sqrt(d))
    aligned = pkv.paged_prefill_varlen(*args)
    buf = torch.zeros(c["q"].numel() + 8, dtype=torch.bfloat16, device=cuda)
    out = buf[8:].view(c["q"].shape)
    assert out.data_ptr() % 32 == 16
    pkv.paged_prefill_varlen(*args, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, aligned)


def test_long_single_sequence_no_cache(cuda):
    pkv = U.lib()
    c = make_case(5, [1000], [0], 8, 2, 128, 256)
    _check_case(pkv, cuda, c, 0.088, use_bt=False)


def test_chunked_walkthrough_equals_oneshot_on_gpu(cuda):
    """600-token prompt, one cached 256-token block, budget 200: the chunk
    [256,456) then [456,600), each stored before the next, matches one call
    over [256,600)."""
    pkv = U.lib()
    bs, hq, hkv, d = 256, 8, 2, 128
    g = torch.Generator().manual_seed(21)
    K = U.bf16_case(g, (600, hkv, d))
    V = U.bf16_case(g, (600, hkv, d))
    Q = U.bf16_case(g, (600, hq, d))
    kc, vc, bt = U.build_paged_cache([K[:256]], [V[:256]], bs, 5, g, extra_blocks_per_seq=[3])
    kc, vc = kc.to(cuda), vc.to(cuda)
    table = bt[0].tolist()
    one = _prefill(pkv, cuda, Q[256:], K[256:], V[256:], kc, vc,
                   torch.tensor([0, 344], dtype=torch.int32),
                   torch.tensor([0, 600], dtype=torch.int32), bt, 0.09, 344, 600)
    parts = []
    for lo, hi in ((256, 456), (456, 600)):
        parts.append(_prefill(pkv, cuda, Q[lo:hi], K[lo:hi], V[lo:hi], kc, vc,
                              torch.tensor([0, hi - lo], dtype=torch.int32),
                              torch.tensor([0, hi], dtype=torch.int32), bt, 0.09, hi - lo, hi))
        slots = torch.tensor([table[p // bs] * bs + p % bs for p in range(lo, hi)],
                             dtype=torch.int32)
        pkv.kv_store(K[lo:hi].to(cuda), V[lo:hi].to(cuda), kc, vc, slots.to(cuda))
    chunked = torch.cat(parts)
    ref = oatt.paged_prefill_varlen(U.f64(Q[256:]), U.f64(K[256:]), U.f64(V[256:]),
                                    kc.cpu(), vc.cpu(), [0, 344], [0, 600], bt.numpy(), 0.09)
    U.assert_close(U.f64(one), ref, "one-shot")
    U.assert_close(U.f64(chunked), ref, "chunked")


# block size 256: cached tiles as TMA boxes; 16: the same prompts (prefixes of
# up to 1024 keys) with every cached tile's rows gathered by cp.async
@pytest.mark.parametrize("bs", [256, 16])
def test_prefill_8b_steps_sampled_rows(cuda, bs):
    pkv = U.lib()
    spec = W.PREFILL_8B
    if bs != spec.block_size:
        spec = dataclasses.replace(spec, block_size=bs, max_cached_blocks=1024 // bs)
    w = W.prefill_workload(spec)
    kc, vc = w.k_cache0.to(cuda), w.v_cache0.to(cuda)
    okc, ovc = U.bits(w.k_cache0), U.bits(w.v_cache0)
    rng = np.random.default_rng(0)
    st = pkv.new_status(cuda)
    for si, step in enumerate(w.steps):
        pkv.kv_store(step.k.to(cuda), step.v.to(cuda), kc, vc, step.slot_mapping.to(cuda),
                     status=st)
        out = pkv.paged_prefill_varlen(step.q.to(cuda), step.k.to(cuda), step.v.to(cuda), kc,
                                       vc, step.cu_seqlens_q.to(cuda),
                                       step.cu_seqlens_k.to(cuda), step.max_seqlen_q,
                                       step.max_seqlen_k, step.block_tables.to(cuda), w.scale,
                                       status=st)
        cu_q = step.cu_seqlens_q.numpy()
        cu_k = step.cu_seqlens_k.numpy()
        rows = {}
        for b in range(len(cu_q) - 1):
            n = int(cu_q[b + 1] - cu_q[b])
            c = int(cu_k[b + 1] - cu_k[b]) - n          # keys already cached
            pick = {0, n - 1, n // 2} | set(rng.integers(0, n, size=5).tolist())
            # both sides of every 128-row query tile boundary (the kernel's
            # work item), and the rows whose position ends a 128-key tile of
            # the cached prefix or starts the next (the partial cached tile's
            # mask and the first tile of the chunk's own keys)
            pick |= {i for t in range(128, n, 128) for i in (t - 1, t)}
            pick |= {i for i in range(n) if (c + i) % 128 in (0, 127)}
            rows[b] = sorted(i for i in pick if 0 <= i < n)
        ref = oatt.paged_prefill_varlen(U.f64(step.q), U.f64(step.k), U.f64(step.v),
                                        torch.from_numpy(okc).view(torch.bfloat16),
                                        torch.from_numpy(ovc).view(torch.bfloat16),
                                        cu_q, step.cu_seqlens_k.numpy(),
                                        step.block_tables.numpy(), w.scale, rows=rows)
        mask = ~np.isnan(ref[:, 0, 0])
        err, rel = U.assert_close(U.f64(out)[mask], ref[mask], f"prefill-8b step {si}")
        print(f"prefill-8b step {si}: {mask.sum()} rows, max abs {err:.3g}, rel L2 {rel:.3g}")
        okc, ovc, _ = okv.kv_store(U.bits(step.k), U.bits(step.v), okc, ovc,
                                   step.slot_mapping.numpy())
    assert U.status_word(st) == 0


def test_inconsistent_seqlens_are_reported(cuda):
    pkv = U.lib()
    c = make_case(8, [10, 12], [0, 0], 2, 1, 64, 16)
    c["cu_k"] = torch.tensor([0, 5, 17], dtype=torch.int32)   # sequence 0: Lk < Lq
    st = pkv.new_status(cuda)
    out = _prefill(pkv, cuda, c["q"], c["k"], c["v"], None, None, c["cu_q"], c["cu_k"], None,
                   0.1, 12, 12, status=st)
    assert U.status_word(st) & pkv.STATUS["BAD_SEQLENS"]
    ref = oatt.paged_prefill_varlen(U.f64(c["q"][10:]), U.f64(c["k"][10:]), U.f64(c["v"][10:]),
                                    None, None, [0, 12], [0, 12], None, 0.1)
    U.assert_close(U.f64(out)[10:], ref, "valid sequence")
