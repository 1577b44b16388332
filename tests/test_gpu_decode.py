"""paged_decode on the GPU against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from oracle import kv_store as okv
from paged_kv_attention_scatter_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode(pkv, w, dev, seqs=None, status_expect=0, max_ctx=None, heads=None):
    st = pkv.new_status(dev)
    out = pkv.paged_decode(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                           w.block_tables.to(dev), w.context_lens.to(dev), w.scale,
                           max_ctx if max_ctx is not None else w.max_context_len, status=st)
    assert U.status_word(st) == status_expect
    kc = w.k_cache.cpu() if w.k_cache.is_cuda else w.k_cache
    vc = w.v_cache.cpu() if w.v_cache.is_cuda else w.v_cache
    ref = oatt.paged_decode(U.f64(w.q), kc, vc, w.block_tables.numpy(),
                            w.context_lens.numpy(), w.scale, seqs=seqs, heads=heads)
    got = U.f64(out)
    idx = list(range(w.q.shape[0])) if seqs is None else list(seqs)
    if heads is None:
        return U.assert_close(got[idx], ref[idx], w.spec.name)
    pairs = [(b, h) for b in idx for h in heads(b)]
    bi, hi = np.array([p[0] for p in pairs]), np.array([p[1] for p in pairs])
    return U.assert_close(got[bi, hi], ref[bi, hi], w.spec.name)


def one_head_per_group(hq, hkv):
    """q heads to check for sequence b: one per kv head, rotating through the
    group with b, so that across sequences every q head is checked."""
    g = hq // hkv
    return lambda b: [kvh * g + (b + kvh) % g for kvh in range(hkv)]


def test_tiny_decode_steps(cuda):
    pkv = U.lib()
    w = W.tiny_workload()
    kc, vc = U.bits(w.k_cache0), U.bits(w.v_cache0)
    p = w.prefill
    kc, vc, _ = okv.kv_store(U.bits(p.k), U.bits(p.v), kc, vc, p.slot_mapping.numpy())
    for st in w.decode_steps:
        kc, vc, _ = okv.kv_store(U.bits(st.k_new), U.bits(st.v_new), kc, vc,
                                 st.slot_mapping.numpy())
        kt = torch.from_numpy(kc).view(torch.bfloat16)
        vt = torch.from_numpy(vc).view(torch.bfloat16)
        out = pkv.paged_decode(st.q.to(cuda), kt.to(cuda), vt.to(cuda),
                               st.block_tables.to(cuda), st.context_lens.to(cuda), w.scale,
                               int(st.context_lens.max()))
        ref = oatt.paged_decode(U.f64(st.q), kt, vt, st.block_tables.numpy(),
                                st.context_lens.numpy(), w.scale)
        U.assert_close(U.f64(out), ref, "tiny decode")


def test_decode_0p6b_full_batch(cuda):
    pkv = U.lib()
    w = W.decode_workload(W.DECODE_0P6B)
    err, rel = _decode(pkv, w, cuda)
    print(f"decode-0.6b: max abs {err:.3g}, rel L2 {rel:.3g}")


def test_decode_32b_every_sequence(cuda):
    """All 256 sequences (contexts 128..32768, so every split/merge case of the
    long rows), one q head per kv head each; the shortest and longest three
    sequences with all 64 q heads."""
    pkv = U.lib()
    w = W.decode_workload(W.DECODE_32B, device=cuda)
    spec = W.DECODE_32B
    err, rel = _decode(pkv, w, cuda, heads=one_head_per_group(spec.num_q_heads,
                                                              spec.num_kv_heads))
    print(f"decode-32b all sequences: max abs {err:.3g}, rel L2 {rel:.3g}")
    order = np.argsort(w.context_lens.numpy())
    seqs = sorted(set(order[:3].tolist() + order[-3:].tolist()))
    err, rel = _decode(pkv, w, cuda, seqs=seqs)
    print(f"decode-32b all heads of {seqs}: max abs {err:.3g}, rel L2 {rel:.3g}")


def test_step_8b_store_then_decode_every_sequence(cuda):
    """All 512 sequences of the step, one q head per kv head each (rotating),
    after the step's kv_store wrote their newest token."""
    pkv = U.lib()
    w = W.decode_workload(W.STEP_8B, device=cuda)
    st = pkv.new_status(cuda)
    kc, vc = w.k_cache, w.v_cache
    seqs = list(range(W.STEP_8B.batch))
    heads = one_head_per_group(W.STEP_8B.num_q_heads, W.STEP_8B.num_kv_heads)
    # oracle-side cache: the sequences' blocks before the step, then the store
    kc_cpu, vc_cpu = kc.cpu(), vc.cpu()
    pkv.kv_store(w.k_new, w.v_new, kc, vc, w.slot_mapping.to(cuda), status=st)
    out = pkv.paged_decode(w.q, kc, vc, w.block_tables.to(cuda), w.context_lens.to(cuda),
                           w.scale, w.max_context_len, status=st)
    assert U.status_word(st) == 0
    ok, ov, _ = okv.kv_store(U.bits(w.k_new), U.bits(w.v_new), U.bits(kc_cpu), U.bits(vc_cpu),
                             w.slot_mapping.numpy())
    ref = oatt.paged_decode(U.f64(w.q), torch.from_numpy(ok).view(torch.bfloat16),
                            torch.from_numpy(ov).view(torch.bfloat16), w.block_tables.numpy(),
                            w.context_lens.numpy(), w.scale, seqs=seqs, heads=heads)
    bi = np.repeat(np.array(seqs), W.STEP_8B.num_kv_heads)
    hi = np.array([h for b in seqs for h in heads(b)])
    err, rel = U.assert_close(U.f64(out)[bi, hi], ref[bi, hi], "step-8b decode")
    print(f"step-8b all sequences: max abs {err:.3g}, rel L2 {rel:.3g}")


# block sizes that are multiples of 64 run the TMA-fed split kernel, the others
# the register-load one; 16 q heads per kv head make two head groups per unit
@pytest.mark.parametrize("hq,hkv,d,bs", [(4, 4, 128, 16), (16, 1, 128, 256), (8, 2, 64, 4),
                                         (6, 2, 64, 32), (12, 4, 128, 64), (16, 1, 64, 64),
                                         (8, 8, 64, 128), (32, 2, 128, 128)])
def test_shapes_and_block_sizes(cuda, hq, hkv, d, bs):
    pkv = U.lib()
    spec = W.DecodeSpec(f"shape {hq}/{hkv}x{d} bs{bs}", seed=hq * 31 + bs, batch=7,
                        num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                        ctx_lo=1, ctx_hi=700)
    w = W.decode_workload(spec)
    _decode(pkv, w, cuda)


@pytest.mark.parametrize("bs", [16, 64])
def test_zero_and_one_key_contexts(cuda, bs):
    pkv = U.lib()
    spec = W.DecodeSpec("edge", seed=9, batch=5, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        block_size=bs, ctx_lo=1, ctx_hi=40)
    w = W.decode_workload(spec)
    w.context_lens[0] = 0
    w.context_lens[1] = 1
    _decode(pkv, w, cuda)


def test_context_over_stated_maximum_is_reported(cuda):
    pkv = U.lib()
    spec = W.DecodeSpec("over", seed=10, batch=4, num_q_heads=4, num_kv_heads=2, head_dim=64,
                        block_size=16, ctx_lo=20, ctx_hi=60)
    w = W.decode_workload(spec)
    st = pkv.new_status(cuda)
    lim = int(w.context_lens.min())
    out = pkv.paged_decode(w.q.to(cuda), w.k_cache.to(cuda), w.v_cache.to(cuda),
                           w.block_tables.to(cuda), w.context_lens.to(cuda), w.scale, lim,
                           status=st)
    assert U.status_word(st) == pkv.STATUS["BAD_CONTEXT_LEN"]
    over = (w.context_lens > lim).nonzero().flatten().tolist()
    assert over and float(out[over].abs().max()) == 0.0


@pytest.mark.parametrize("bs", [16, 64])
def test_bad_block_id_is_reported_not_read(cuda, bs):
    pkv = U.lib()
    spec = W.DecodeSpec("badblk", seed=12, batch=3, num_q_heads=4, num_kv_heads=1,
                        head_dim=128, block_size=bs, ctx_lo=2 * bs + 8, ctx_hi=4 * bs - 4)
    w = W.decode_workload(spec)
    w.block_tables[1, 1] = 10_000_000
    st = pkv.new_status(cuda)
    out = pkv.paged_decode(w.q.to(cuda), w.k_cache.to(cuda), w.v_cache.to(cuda),
                           w.block_tables.to(cuda), w.context_lens.to(cuda), w.scale,
                           w.max_context_len, status=st)
    assert U.status_word(st) == pkv.STATUS["BAD_BLOCK_ID"]
    assert torch.isfinite(out.float()).all()
    ref = oatt.paged_decode(U.f64(w.q), w.k_cache, w.v_cache, w.block_tables.numpy(),
                            w.context_lens.numpy(), w.scale, seqs=[0, 2])
    U.assert_close(U.f64(out)[[0, 2]], ref[[0, 2]], "unaffected sequences")


def test_workspace_too_small_is_rejected(cuda):
    pkv = U.lib()
    w = W.decode_workload(W.DecodeSpec("ws", seed=1, batch=2, num_q_heads=2, num_kv_heads=1,
                                       head_dim=64, block_size=16, ctx_lo=5, ctx_hi=9))
    ws = torch.empty(16, dtype=torch.uint8, device=cuda)
    with pytest.raises(RuntimeError, match="workspace"):
        pkv.paged_decode(w.q.to(cuda), w.k_cache.to(cuda), w.v_cache.to(cuda),
                         w.block_tables.to(cuda), w.context_lens.to(cuda), w.scale,
                         w.max_context_len, workspace=ws)


@pytest.mark.parametrize("max_ctx_scale", [1, 64])
def test_stated_maximum_context_sets_the_chunking(cuda, max_ctx_scale):
    """The chunk size comes from the stated maximum context alone: the exact
    maximum gives 64-key chunks (up to 15 per sequence), a 64x larger one
    1024-key chunks.  Both chunkings must match the oracle."""
    pkv = U.lib()
    spec = W.DecodeSpec("merge", seed=77, batch=24, num_q_heads=8, num_kv_heads=4, head_dim=128,
                        block_size=64, ctx_lo=1, ctx_hi=900)
    w = W.decode_workload(spec)
    max_ctx = int(w.context_lens.max()) * max_ctx_scale
    bt_cols = -(-max_ctx // spec.block_size)
    bt = torch.full((spec.batch, bt_cols), -1, dtype=torch.int32)
    bt[:, :w.block_tables.shape[1]] = w.block_tables
    st = pkv.new_status(cuda)
    out = pkv.paged_decode(w.q.to(cuda), w.k_cache.to(cuda), w.v_cache.to(cuda), bt.to(cuda),
                           w.context_lens.to(cuda), w.scale, max_ctx, status=st)
    assert U.status_word(st) == 0
    ref = oatt.paged_decode(U.f64(w.q), w.k_cache, w.v_cache, w.block_tables.numpy(),
                            w.context_lens.numpy(), w.scale)
    U.assert_close(U.f64(out), ref, f"decode, max_ctx x{max_ctx_scale}")


def test_decode_0p6b_plan_and_layer_runs_in_a_graph(cuda):
    """The headline's launch configuration at full size: one plan, then one run
    per layer of a [2, L, NB, bs, Hkv, D] pool, all captured in one CUDA graph
    and replayed.  Each layer holds its own random cache; every layer's output
    is checked against the float64 oracle on a sample of sequences (the
    shortest, the longest and a spread between)."""
    pkv = U.lib()
    spec = W.DECODE_0P6B
    w = W.decode_workload(spec)
    L = 3
    g = torch.Generator().manual_seed(404)
    pool = torch.empty((2, L) + tuple(w.k_cache.shape), dtype=torch.bfloat16)
    for layer in range(L):
        pool[0, layer] = torch.randn(w.k_cache.shape, generator=g).to(torch.bfloat16)
        pool[1, layer] = torch.randn(w.v_cache.shape, generator=g).to(torch.bfloat16)
    pool_d = pool.to(cuda)
    layers = [pkv.layer_cache(pool_d, layer) for layer in range(L)]
    q, bt, ctx = w.q.to(cuda), w.block_tables.to(cuda), w.context_lens.to(cuda)
    mc, mb = w.max_context_len, bt.shape[1]
    ws = torch.empty(pkv.paged_decode_workspace_bytes(spec.batch, spec.num_q_heads, mc,
                                                      layers[0][0]),
                     dtype=torch.uint8, device=cuda)
    outs = [torch.zeros_like(q) for _ in range(L)]
    st = pkv.new_status(cuda)

    def step():
        pkv.paged_decode_plan(ctx, spec.num_q_heads, mc, mb, layers[0][0], workspace=ws,
                              status=st)
        for (kc, vc), o in zip(layers, outs):
            pkv.paged_decode_run(q, kc, vc, bt, ctx, w.scale, mc, ws, out=o, status=st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for o in outs:
        o.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert U.status_word(st) == 0
    order = np.argsort(w.context_lens.numpy())
    seqs = sorted(set([int(order[0]), int(order[-1])] + [int(x) for x in order[::9]]))
    for layer in range(L):
        ref = oatt.paged_decode(U.f64(w.q), pool[0, layer], pool[1, layer],
                                w.block_tables.numpy(), w.context_lens.numpy(), w.scale,
                                seqs=seqs)
        U.assert_close(U.f64(outs[layer])[seqs], ref[seqs], f"decode-0.6b layer {layer}")
