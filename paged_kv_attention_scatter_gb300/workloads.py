"""Seeded synthetic workloads for the paged-KV hot path.

This module only draws inputs: random tensors, block tables, context lengths,
chunk boundaries and the per-token slot lists a serving engine's host side
would hand to the kernels.  It holds none of the attention or sampling
arithmetic, imports neither the CUDA binding nor the CPU oracle, and serves
both of them.

The shapes follow the five synthetic workloads (Qwen3-shaped attention layers):

  tiny       8 blocks x 4 slots, 2 q heads / 1 kv head, head_dim 64; prompts of
             7 and 11 tokens, prefill, 3 decode steps each, sampler over 1000
  decode-0.6b   B=64, 16/8 heads, D=128, block 256, ctx ~ U[512, 4096]
  prefill-8b    16 prompts L ~ U[1024, 8192], 32/8 heads, D=128, block 256,
                0..4 shared cached prefix blocks, 16384-token chunks
  decode-32b    B=256, 64/8 heads, ctx log-uniform in [128, 32768], pool 7000
  step-8b       B=512, 32/8 heads, ctx ~ U[256, 8192]; kv_store of the new
                token, decode, sampler over vocab 151936
  mixed-8b      a continuous-batching step: 256 decode rows (ctx ~ U[256, 8192])
                and 4 prefill chunks in one varlen batch, 32/8 heads

Conventions (all choices of the input recipe, not of the method):
  * workload n uses seed n-1; integer draws are inclusive-uniform;
  * Q/K/V are torch.randn fp32 rounded to bf16;
  * every cache slot that holds no token is bf16 NaN, so a stray read of it
    shows up in the outputs;
  * block_tables are int32, padded with -1 past a sequence's last block;
  * Exp(1) noise is E = -ln(U) with U uniform in (0, 1].

How the engine-side metadata is formed (a slot is block_id*block_size + offset
inside the block; a sequence's blocks come from its block table in order; a
new block is appended only when the last one is full) mirrors the host code the
pages describe ("一个 prompt 的一生" §3.3.2 and §4; "《Nano-vLLM源码逐行解析》第2篇"
sequence.py block counters).  The tests check these lists against the oracle's
independent restatement.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN = float("nan")


# ----------------------------------------------------------------------------
# workload descriptions
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class DecodeSpec:
    name: str
    seed: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    ctx_lo: int
    ctx_hi: int
    ctx_dist: str = "uniform"          # "uniform" (integers) or "loguniform"
    num_blocks: int | None = None      # None: pool sized to fit exactly
    store_new_token: bool = False      # the step writes the token at ctx-1 first
    vocab: int | None = None           # sampler vocabulary (None: no sampler)
    logit_sigma: float = 3.0
    logit_spikes: int = 0
    t_lo: float = 1.0
    t_hi: float = 1.0


@dataclass(frozen=True)
class PrefillSpec:
    name: str
    seed: int
    num_prompts: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    len_lo: int
    len_hi: int
    max_cached_blocks: int             # prompt r has k_r ~ U{0..max} shared blocks
    token_budget: int                  # new tokens per chunked step
    first_only_chunking: bool = False  # the pages' scheduler rule (kept as a flag)
    spare_blocks: int = 0


DECODE_0P6B = DecodeSpec("decode-0.6b B=64 16/8x128 bs256 ctx U[512,4096]", seed=1,
                         batch=64, num_q_heads=16, num_kv_heads=8, head_dim=128,
                         block_size=256, ctx_lo=512, ctx_hi=4096)
PREFILL_8B = PrefillSpec("prefill-8b 16 prompts U[1024,8192] 32/8x128 bs256 "
                         "prefix 0..4 blocks budget 16384", seed=2,
                         num_prompts=16, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, block_size=256, len_lo=1024, len_hi=8192,
                         max_cached_blocks=4, token_budget=16384)
DECODE_32B = DecodeSpec("decode-32b B=256 64/8x128 bs256 ctx logU[128,32768] NB=7000",
                        seed=3, batch=256, num_q_heads=64, num_kv_heads=8,
                        head_dim=128, block_size=256, ctx_lo=128, ctx_hi=32768,
                        ctx_dist="loguniform", num_blocks=7000)
STEP_8B = DecodeSpec("step-8b B=512 32/8x128 bs256 ctx U[256,8192] V=151936",
                     seed=4, batch=512, num_q_heads=32, num_kv_heads=8,
                     head_dim=128, block_size=256, ctx_lo=256, ctx_hi=8192,
                     store_new_token=True, vocab=151936, logit_sigma=3.0,
                     logit_spikes=4, t_lo=0.2, t_hi=1.2)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32,
                       device=device).to(torch.bfloat16)


def randint_incl(lo: int, hi: int, n: int, gen: torch.Generator) -> list[int]:
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def slot_list(block_table, block_size: int, start: int, count: int) -> list[int]:
    """Slots of logical token positions [start, start+count) of one sequence."""
    out = []
    for pos in range(start, start + count):
        out.append(block_table[pos // block_size] * block_size + pos % block_size)
    return out


def pad_tables(tables: list[list[int]], width: int | None = None) -> torch.Tensor:
    width = max((len(t) for t in tables), default=0) if width is None else width
    width = max(width, 1)
    bt = torch.full((len(tables), width), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        if t:
            bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return bt


def fill_pool(num_blocks: int, block_size: int, hkv: int, d: int,
              valid: list[tuple[int, int]], gen_dev: torch.Generator,
              device) -> torch.Tensor:
    """A [NB, bs, Hkv, D] bf16 pool: random rows at `valid` (block, rows_used)
    entries, NaN everywhere else."""
    pool = randn_bf16((num_blocks, block_size, hkv, d), gen_dev, device)
    mask = torch.zeros(num_blocks, block_size, dtype=torch.bool)
    for blk, used in valid:
        mask[blk, :used] = True
    pool[~mask.to(device)] = BF16_NAN
    return pool


# ----------------------------------------------------------------------------
# decode workloads (decode-0.6b, decode-32b, step-8b)
# ----------------------------------------------------------------------------
def draw_context_lens(spec: DecodeSpec, gen: torch.Generator) -> list[int]:
    if spec.ctx_dist == "uniform":
        return randint_incl(spec.ctx_lo, spec.ctx_hi, spec.batch, gen)
    if spec.ctx_dist == "loguniform":
        u = torch.rand(spec.batch, generator=gen, dtype=torch.float64)
        lo, hi = math.log(spec.ctx_lo), math.log(spec.ctx_hi)
        return [max(spec.ctx_lo, min(spec.ctx_hi, int(math.floor(math.exp(lo + (hi - lo) * x)))))
                for x in u.tolist()]
    raise ValueError(spec.ctx_dist)


@dataclass
class DecodeWorkload:
    spec: DecodeSpec
    context_lens: torch.Tensor      # (B,) int32: keys attended, incl. the new token
    block_tables: torch.Tensor      # (B, MB) int32, -1 padded
    q: torch.Tensor                 # (B, Hq, D) bf16
    k_cache: torch.Tensor           # (NB, bs, Hkv, D) bf16
    v_cache: torch.Tensor
    scale: float
    max_context_len: int
    # only when the step stores the new token first
    k_new: torch.Tensor | None = None       # (B, Hkv, D) bf16
    v_new: torch.Tensor | None = None
    slot_mapping: torch.Tensor | None = None  # (B,) int32
    # only when the step samples
    logits: torch.Tensor | None = None        # (B, V) fp32
    temperatures: torch.Tensor | None = None  # (B,) fp32
    exp_noise: torch.Tensor | None = None     # (B, V) fp32

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]


def decode_workload(spec: DecodeSpec, device="cpu") -> DecodeWorkload:
    """Builds one decode step.  Integer draws on a CPU generator; the big random
    tensors on a generator of `device` (seeded with the same seed)."""
    g = _gen(spec.seed)
    gdev = _gen(spec.seed, device)
    bs = spec.block_size
    ctx = draw_context_lens(spec, g)
    need = [ceil_div(c, bs) for c in ctx]
    nb = spec.num_blocks if spec.num_blocks is not None else sum(need)
    if nb < sum(need):
        raise ValueError("pool too small for the drawn contexts")
    perm = torch.randperm(nb, generator=g).tolist()
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n])
        at += n
    # tokens already in the cache before the step: ctx-1 if the step stores
    # the new token itself, else all ctx
    held = [c - 1 if spec.store_new_token else c for c in ctx]
    valid = []
    for t, h in zip(tables, held):
        for i, blk in enumerate(t):
            used = min(bs, h - i * bs)
            if used > 0:
                valid.append((blk, used))
    hkv, d = spec.num_kv_heads, spec.head_dim
    k_cache = fill_pool(nb, bs, hkv, d, valid, gdev, device)
    v_cache = fill_pool(nb, bs, hkv, d, valid, gdev, device)
    q = randn_bf16((spec.batch, spec.num_q_heads, d), gdev, device)
    w = DecodeWorkload(spec=spec,
                       context_lens=torch.tensor(ctx, dtype=torch.int32),
                       block_tables=pad_tables(tables), q=q,
                       k_cache=k_cache, v_cache=v_cache,
                       scale=1.0 / math.sqrt(d), max_context_len=max(ctx))
    if spec.store_new_token:
        w.k_new = randn_bf16((spec.batch, hkv, d), gdev, device)
        w.v_new = randn_bf16((spec.batch, hkv, d), gdev, device)
        w.slot_mapping = torch.tensor(
            [slot_list(t, bs, c - 1, 1)[0] for t, c in zip(tables, ctx)],
            dtype=torch.int32)
    if spec.vocab is not None:
        s = sampler_inputs(spec.batch, spec.vocab, spec.logit_sigma,
                           spec.logit_spikes, spec.t_lo, spec.t_hi, g)
        w.logits, w.temperatures, w.exp_noise = s
    return w


def sampler_inputs(batch: int, vocab: int, sigma: float, spikes: int,
                   t_lo: float, t_hi: float, gen: torch.Generator):
    """fp32 logits ~ N(0, sigma) with `spikes` distinct entries per row raised
    by +10, temperatures ~ U[t_lo, t_hi], and Exp(1) noise E = -ln(U)."""
    logits = torch.randn((batch, vocab), generator=gen, dtype=torch.float32) * sigma
    for r in range(batch):
        if spikes:
            idx: list[int] = []
            while len(idx) < spikes:                 # distinct indices per row
                i = int(torch.randint(0, vocab, (1,), generator=gen))
                if i not in idx:
                    idx.append(i)
            logits[r, idx] += 10.0
    temps = (t_lo + (t_hi - t_lo) * torch.rand(batch, generator=gen,
                                               dtype=torch.float32)).float()
    u = 1.0 - torch.rand((batch, vocab), generator=gen, dtype=torch.float32)
    noise = -torch.log(u)
    return logits, temps, noise


# ----------------------------------------------------------------------------
# chunked, prefix-cached prefill (prefill-8b)
# ----------------------------------------------------------------------------
@dataclass
class PrefillStep:
    q: torch.Tensor                 # (Tq, Hq, D) bf16 -- queries of this chunk
    k: torch.Tensor                 # (Tq, Hkv, D) bf16 -- the chunk's own K/V
    v: torch.Tensor
    cu_seqlens_q: torch.Tensor      # (B+1,) int32
    cu_seqlens_k: torch.Tensor      # (B+1,) int32
    block_tables: torch.Tensor      # (B, MB) int32
    slot_mapping: torch.Tensor      # (Tq,) int32
    seq_ids: list[int]              # prompt index of each sequence in the step
    q_start: list[int]              # first query position of each sequence
    max_seqlen_q: int
    max_seqlen_k: int


@dataclass
class PrefillWorkload:
    spec: PrefillSpec
    prompt_lens: list[int]
    cached_blocks: list[int]        # k_r
    block_tables: list[list[int]]   # per prompt, full length
    k_cache0: torch.Tensor          # pool before the first step (prefix filled)
    v_cache0: torch.Tensor
    steps: list[PrefillStep]
    scale: float

    @property
    def num_blocks(self) -> int:
        return self.k_cache0.shape[0]


def chunk_plan(lens_new: list[int], budget: int, first_only: bool):
    """Splits per-prompt new-token counts into steps of `budget` tokens in
    prompt order.  Each step is a list of (prompt, start_offset, count)."""
    steps, cur, room = [], [], budget
    for r, n in enumerate(lens_new):
        off = 0
        while off < n:
            if room == 0 or (first_only and cur and n - off > room):
                steps.append(cur)
                cur, room = [], budget
            take = min(room, n - off)
            cur.append((r, off, take))
            off += take
            room -= take
    if cur:
        steps.append(cur)
    return steps


def prefill_workload(spec: PrefillSpec, device="cpu",
                     prompt_lens: list[int] | None = None,
                     cached_blocks: list[int] | None = None) -> PrefillWorkload:
    g = _gen(spec.seed)
    gdev = _gen(spec.seed, device)
    bs, hq, hkv, d = spec.block_size, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    P = spec.num_prompts
    if prompt_lens is None:
        prompt_lens = randint_incl(spec.len_lo, spec.len_hi, P, g)
    if cached_blocks is None:
        cached_blocks = randint_incl(0, spec.max_cached_blocks, P, g)
    # never cache a whole prompt: at least one token is computed
    cached_blocks = [min(kb, (L - 1) // bs) for kb, L in zip(cached_blocks, prompt_lens)]
    n_prefix = spec.max_cached_blocks
    own = [ceil_div(L, bs) - kb for L, kb in zip(prompt_lens, cached_blocks)]
    nb = n_prefix + sum(own) + spec.spare_blocks
    # the shared prefix blocks are ids 0..n_prefix-1 of a shuffled pool
    perm = torch.randperm(nb, generator=g).tolist()
    prefix_ids, rest = perm[:n_prefix], perm[n_prefix:]
    tables, at = [], 0
    for kb, n in zip(cached_blocks, own):
        tables.append(prefix_ids[:kb] + rest[at:at + n])
        at += n
    # cache state before the first step: the prefix blocks hold fixed K/V
    valid = [(b, bs) for b in prefix_ids]
    k0 = fill_pool(nb, bs, hkv, d, valid, gdev, device)
    v0 = fill_pool(nb, bs, hkv, d, valid, gdev, device)
    # per-prompt K/V of the new tokens and Q of every computed token
    lens_new = [L - kb * bs for L, kb in zip(prompt_lens, cached_blocks)]
    qs = [randn_bf16((n, hq, d), gdev, device) for n in lens_new]
    ks = [randn_bf16((n, hkv, d), gdev, device) for n in lens_new]
    vs = [randn_bf16((n, hkv, d), gdev, device) for n in lens_new]
    steps = []
    for plan in chunk_plan(lens_new, spec.token_budget, spec.first_only_chunking):
        cu_q, cu_k, slots, sid, qst = [0], [0], [], [], []
        q_parts, k_parts, v_parts, bts = [], [], [], []
        for r, off, take in plan:
            c = cached_blocks[r] * bs + off          # tokens already in the cache
            cu_q.append(cu_q[-1] + take)
            cu_k.append(cu_k[-1] + c + take)
            slots += slot_list(tables[r], bs, c, take)
            q_parts.append(qs[r][off:off + take])
            k_parts.append(ks[r][off:off + take])
            v_parts.append(vs[r][off:off + take])
            bts.append(tables[r])
            sid.append(r)
            qst.append(c)
        steps.append(PrefillStep(
            q=torch.cat(q_parts), k=torch.cat(k_parts), v=torch.cat(v_parts),
            cu_seqlens_q=torch.tensor(cu_q, dtype=torch.int32),
            cu_seqlens_k=torch.tensor(cu_k, dtype=torch.int32),
            block_tables=pad_tables(bts), slot_mapping=torch.tensor(slots, dtype=torch.int32),
            seq_ids=sid, q_start=qst,
            max_seqlen_q=max(b - a for a, b in zip(cu_q, cu_q[1:])),
            max_seqlen_k=max(b - a for a, b in zip(cu_k, cu_k[1:]))))
    return PrefillWorkload(spec=spec, prompt_lens=prompt_lens, cached_blocks=cached_blocks,
                           block_tables=tables, k_cache0=k0, v_cache0=v0, steps=steps,
                           scale=1.0 / math.sqrt(d))


# ----------------------------------------------------------------------------
# a continuous-batching step: decode rows and prefill chunks together
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class MixedSpec:
    name: str
    seed: int
    num_decode: int                    # one-query sequences
    num_prefill: int                   # prefill chunks
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    ctx_lo: int                        # decode context, the new token included
    ctx_hi: int
    new_lo: int                        # new tokens of a prefill chunk
    new_hi: int
    cached_lo: int                     # tokens of a chunk's sequence already cached
    cached_hi: int


MIXED_8B = MixedSpec("mixed-8b 256 decode rows ctx U[256,8192] + 4 chunks of U[512,2048] "
                     "new tokens on U[0,4096] cached, 32/8x128 bs256", seed=5,
                     num_decode=256, num_prefill=4, num_q_heads=32, num_kv_heads=8,
                     head_dim=128, block_size=256, ctx_lo=256, ctx_hi=8192,
                     new_lo=512, new_hi=2048, cached_lo=0, cached_hi=4096)


@dataclass
class MixedWorkload:
    spec: MixedSpec
    step: PrefillStep               # the varlen batch, decode rows first
    k_cache0: torch.Tensor          # pool before the step: cached tokens filled
    v_cache0: torch.Tensor
    scale: float


def mixed_workload(spec: MixedSpec, device="cpu") -> MixedWorkload:
    """One step of a batch that mixes decode rows (one new token on ctx-1
    cached ones) with prefill chunks (new tokens on a cached prefix), in one
    varlen batch; every sequence owns its blocks, and the step's slot_mapping
    places each new token at its position in its own block table."""
    g = _gen(spec.seed)
    gdev = _gen(spec.seed, device)
    bs, hq, hkv, d = spec.block_size, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    ctx = randint_incl(spec.ctx_lo, spec.ctx_hi, spec.num_decode, g)
    new = randint_incl(spec.new_lo, spec.new_hi, spec.num_prefill, g)
    cached = randint_incl(spec.cached_lo, spec.cached_hi, spec.num_prefill, g)
    seqs = [(1, c - 1) for c in ctx] + list(zip(new, cached))    # (new, cached)
    need = [ceil_div(n + c, bs) for n, c in seqs]
    nb = sum(need)
    perm = torch.randperm(nb, generator=g).tolist()
    tables, at = [], 0
    for n in need:
        tables.append(perm[at:at + n])
        at += n
    valid = []
    for t, (_, c) in zip(tables, seqs):
        for i, blk in enumerate(t):
            used = min(bs, c - i * bs)
            if used > 0:
                valid.append((blk, used))
    k0 = fill_pool(nb, bs, hkv, d, valid, gdev, device)
    v0 = fill_pool(nb, bs, hkv, d, valid, gdev, device)
    T = sum(n for n, _ in seqs)
    q = randn_bf16((T, hq, d), gdev, device)
    k = randn_bf16((T, hkv, d), gdev, device)
    v = randn_bf16((T, hkv, d), gdev, device)
    cu_q, cu_k, slots = [0], [0], []
    for t, (n, c) in zip(tables, seqs):
        cu_q.append(cu_q[-1] + n)
        cu_k.append(cu_k[-1] + c + n)
        slots += slot_list(t, bs, c, n)
    step = PrefillStep(q=q, k=k, v=v, cu_seqlens_q=torch.tensor(cu_q, dtype=torch.int32),
                       cu_seqlens_k=torch.tensor(cu_k, dtype=torch.int32),
                       block_tables=pad_tables(tables),
                       slot_mapping=torch.tensor(slots, dtype=torch.int32),
                       seq_ids=list(range(len(seqs))), q_start=[c for _, c in seqs],
                       max_seqlen_q=max(n for n, _ in seqs),
                       max_seqlen_k=max(n + c for n, c in seqs))
    return MixedWorkload(spec=spec, step=step, k_cache0=k0, v_cache0=v0,
                         scale=1.0 / math.sqrt(d))


# ----------------------------------------------------------------------------
# tiny end-to-end scenario
# ----------------------------------------------------------------------------
@dataclass
class TinyDecodeStep:
    q: torch.Tensor                 # (2, Hq, D)
    k_new: torch.Tensor             # (2, Hkv, D)
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # (2,)
    block_tables: torch.Tensor      # (2, MB)
    context_lens: torch.Tensor      # (2,)


@dataclass
class TinyWorkload:
    num_blocks: int
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prefill: PrefillStep
    decode_steps: list[TinyDecodeStep]
    logits: torch.Tensor
    temperatures: torch.Tensor
    exp_noise: torch.Tensor
    scale: float
    k_cache0: torch.Tensor
    v_cache0: torch.Tensor
    block_tables_final: list[list[int]] = field(default_factory=list)


def tiny_workload(seed: int = 0) -> TinyWorkload:
    """8 blocks of 4 slots, GQA 2:1, D=64; prompts of 7 and 11 tokens; then three
    decode steps per sequence with a block appended when the last one is full;
    finally one sampler call over a 1000-entry vocabulary."""
    g = _gen(seed)
    nb, bs, hq, hkv, d = 8, 4, 2, 1, 64
    perm = torch.randperm(nb, generator=g).tolist()
    lens = [7, 11]
    tables = [perm[0:2], perm[2:5]]
    free = perm[5:]
    k0 = torch.full((nb, bs, hkv, d), BF16_NAN, dtype=torch.bfloat16)
    v0 = k0.clone()
    q = randn_bf16((sum(lens), hq, d), g)
    k = randn_bf16((sum(lens), hkv, d), g)
    v = randn_bf16((sum(lens), hkv, d), g)
    slots = slot_list(tables[0], bs, 0, lens[0]) + slot_list(tables[1], bs, 0, lens[1])
    pre = PrefillStep(q=q, k=k, v=v,
                      cu_seqlens_q=torch.tensor([0, 7, 18], dtype=torch.int32),
                      cu_seqlens_k=torch.tensor([0, 7, 18], dtype=torch.int32),
                      block_tables=pad_tables(tables),
                      slot_mapping=torch.tensor(slots, dtype=torch.int32),
                      seq_ids=[0, 1], q_start=[0, 0], max_seqlen_q=11, max_seqlen_k=11)
    steps = []
    n = list(lens)
    for _ in range(3):
        new_slots = []
        for i in range(2):
            n[i] += 1
            if len(tables[i]) * bs < n[i]:           # last block full: append one
                tables[i] = tables[i] + [free.pop(0)]
            new_slots += slot_list(tables[i], bs, n[i] - 1, 1)
        steps.append(TinyDecodeStep(
            q=randn_bf16((2, hq, d), g), k_new=randn_bf16((2, hkv, d), g),
            v_new=randn_bf16((2, hkv, d), g),
            slot_mapping=torch.tensor(new_slots, dtype=torch.int32),
            block_tables=pad_tables(tables), context_lens=torch.tensor(n, dtype=torch.int32)))
    logits, temps, noise = sampler_inputs(2, 1000, 4.0, 0, 0.7, 0.7, g)
    temps = torch.tensor([0.7, 1.0], dtype=torch.float32)
    return TinyWorkload(nb, bs, hq, hkv, d, pre, steps, logits, temps, noise,
                        1.0 / math.sqrt(d), k0, v0, [list(t) for t in tables])
