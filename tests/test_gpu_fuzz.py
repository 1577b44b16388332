"""Seeded random configurations against the float64 oracle.

Each case draws its own kv heads (1, 2, 4, 8), q heads per kv head (1 to 16, so
one or two mma head groups in decode), head_dim (64 or 128), cache block size
(1 to 512: TMA boxes, gathered rows, the register-load decode kernel) and
sequence lengths (empty and one-key contexts included), scatters the logical
K/V through a shuffled pool whose unused slots hold NaN, and compares
paged_decode, paged_prefill_varlen and the mixed store + attention call with
the oracle (the store bit for bit).  The samplers draw their own vocabulary
(1 to 200000 entries, multiples of 4 or not), temperatures and logit spread,
with supplied and in-kernel noise, and must give the oracle's token ids
(any near-top index where float32 and float64 keys may legitimately tie)."""
import numpy as np
import pytest
import torch

import gpu_util as U
from oracle import attention as oatt
from oracle import kv_store as okv
from oracle import sampler as osm
from test_gpu_fused_prefill import _slots
from test_gpu_prefill import _check_case, make_case

pytestmark = pytest.mark.gpu

BLOCK_SIZES = [1, 2, 3, 4, 5, 7, 8, 12, 16, 24, 32, 48, 64, 96, 100, 128, 192, 256, 384, 512]


def _shape(rng):
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    return hkv * g, hkv, int(rng.choice([64, 128])), int(rng.choice(BLOCK_SIZES))


@pytest.mark.parametrize("seed", range(48))
def test_decode_random_configurations(cuda, seed):
    rng = np.random.default_rng(7000 + seed)
    pkv = U.lib()
    hq, hkv, d, bs = _shape(rng)
    B = int(rng.integers(1, 17))
    ctx = rng.integers(2, 2500, size=B)
    ctx[rng.random(B) < 0.15] = 0                    # padded rows write zeros
    ctx[rng.random(B) < 0.15] = 1
    gen = torch.Generator().manual_seed(7000 + seed)
    K = [U.bf16_case(gen, (int(c), hkv, d)) for c in ctx]
    V = [U.bf16_case(gen, (int(c), hkv, d)) for c in ctx]
    nb = int(sum(-(-int(c) // bs) for c in ctx)) + 3
    kc, vc, bt = U.build_paged_cache(K, V, bs, nb, gen)
    q = U.bf16_case(gen, (B, hq, d))
    scale = d ** -0.5
    max_ctx = max(int(ctx.max()), 1)
    st = pkv.new_status(cuda)
    ctx_t = torch.tensor(ctx, dtype=torch.int32)
    out = pkv.paged_decode(q.to(cuda), kc.to(cuda), vc.to(cuda), bt.to(cuda), ctx_t.to(cuda),
                           scale, max_ctx, status=st)
    assert U.status_word(st) == 0
    ref = oatt.paged_decode(U.f64(q), kc, vc, bt.numpy(), ctx, scale)
    U.assert_close(U.f64(out), ref, f"decode {hq}/{hkv}x{d} bs{bs} B={B}")


@pytest.mark.parametrize("seed", range(32))
def test_prefill_random_configurations(cuda, seed):
    rng = np.random.default_rng(8000 + seed)
    pkv = U.lib()
    hq, hkv, d, bs = _shape(rng)
    hq = min(hq, 32)
    hq -= hq % hkv
    B = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(1, 400, size=B)]
    cached = [int(x) for x in rng.integers(0, 1500, size=B)]
    for b in range(B):
        if rng.random() < 0.2:
            cached[b] = 0
        if rng.random() < 0.15:
            lens[b] = 1
    c = make_case(8000 + seed, lens, cached, hq, hkv, d, bs)
    _check_case(pkv, cuda, c, d ** -0.5)


@pytest.mark.parametrize("seed", range(24))
def test_mixed_store_and_attention_random_configurations(cuda, seed):
    rng = np.random.default_rng(9000 + seed)
    pkv = U.lib()
    hq, hkv, d, bs = _shape(rng)
    hq = min(hq, 32)
    hq -= hq % hkv
    B = int(rng.integers(2, 10))
    lens = [1 if rng.random() < 0.6 else int(rng.integers(2, 300)) for _ in range(B)]
    cached = [int(x) for x in rng.integers(0, 1200, size=B)]
    c = make_case(9000 + seed, lens, cached, hq, hkv, d, bs)
    sl = _slots(c, lens, cached, bs)
    kc, vc = c["kc"].to(cuda), c["vc"].to(cuda)
    st = pkv.new_status(cuda)
    scale = d ** -0.5
    out = pkv.kv_store_paged_attention_varlen(c["q"].to(cuda), c["k"].to(cuda), c["v"].to(cuda),
                                              kc, vc, sl.to(cuda), c["cu_q"].to(cuda),
                                              c["cu_k"].to(cuda), c["max_sq"], c["max_sk"],
                                              c["bt"].to(cuda), scale, status=st)
    assert U.status_word(st) == 0
    # the store, bit for bit
    ok_, ov_, _ = okv.kv_store(U.bits(c["k"]), U.bits(c["v"]), U.bits(c["kc"]), U.bits(c["vc"]),
                               sl.numpy())
    assert np.array_equal(U.bits(kc), ok_) and np.array_equal(U.bits(vc), ov_)
    # the attention of every row (the new keys come from k/v in the oracle)
    ref = oatt.paged_prefill_varlen(U.f64(c["q"]), U.f64(c["k"]), U.f64(c["v"]), c["kc"],
                                    c["vc"], c["cu_q"].numpy(), c["cu_k"].numpy(),
                                    c["bt"].numpy(), scale)
    U.assert_close(U.f64(out), ref, f"mixed {hq}/{hkv}x{d} bs{bs} lens={lens}")


def _ids_match(ids, ref, bad, keys):
    near = osm.near_ties(keys)
    for r in range(len(ids)):
        if r in bad:
            assert ids[r] == 0
        else:
            assert ids[r] == ref[r] or (len(near[r]) > 1 and ids[r] in near[r]), \
                (r, ids[r], ref[r], near[r])


@pytest.mark.parametrize("seed", range(24))
def test_samplers_random_configurations(cuda, seed):
    rng = np.random.default_rng(10000 + seed)
    pkv = U.lib()
    B = int(rng.integers(1, 40))
    vocab = int(rng.choice([1, 2, 3, 5, 7, 64, 1000, 4097, 32000, 50257, 151936, 200000]))
    sigma = float(rng.choice([0.5, 3.0, 12.0]))
    g = torch.Generator().manual_seed(10000 + seed)
    logits = torch.randn((B, vocab), generator=g, dtype=torch.float32) * sigma
    temps = torch.from_numpy(rng.uniform(0.05, 2.0, size=B).astype(np.float32))
    noise = -torch.log(1.0 - torch.rand((B, vocab), generator=g, dtype=torch.float32))
    # supplied noise
    ids = pkv.sample(logits.to(cuda), temps.to(cuda), noise.to(cuda)).cpu().numpy()
    ref, bad = osm.sample(logits.numpy(), temps.numpy(), noise.numpy())
    _, keys = osm.sample_key_form(logits.numpy(), temps.numpy(), noise.numpy())
    _ids_match(ids, ref, bad, keys)
    # noise drawn in the kernel from Philox4x32-10
    seed_p, offset = int(rng.integers(0, 2**63)), int(rng.integers(0, 2**40))
    ids = pkv.sample_philox(logits.to(cuda), temps.to(cuda), seed_p, offset).cpu().numpy()
    ref, bad = osm.sample_philox(logits.numpy(), temps.numpy(), seed_p, offset)
    E = osm.philox_exp_noise(B, vocab, seed_p, offset)
    _, keys = osm.sample_key_form(logits.numpy(), temps.numpy(), E)
    _ids_match(ids, ref, bad, keys)
